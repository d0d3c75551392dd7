"""Seeded, counter-based synthetic inputs (see synth.h for the definition).

This module makes inputs only; it holds none of the shard-local step's
arithmetic. The CPU oracle's tests and the CUDA path's tests and bench both
draw from it, so both sides see identical bits. The host fill and the device
fill produce the same values for the same arguments.

Streams: MASTER draws the fp32 master weights, GRAD the incoming gradient
slices (``rank`` = source rank, ``step`` = optimizer step), OUTLIER selects
the scaled gradient entries of the outlier workload. ``index`` is always the
global flat index, so values do not depend on the sharding.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzs_synth.so")

STREAM_MASTER = 1
STREAM_GRAD = 2
STREAM_OUTLIER = 3

_SOURCES = ["synth_host.c", "synth_dev.cu"]


def build_command():
    return [
        "nvcc", "-shared", "-O2", "-std=c++17",
        "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
        "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
        "-Xcompiler", "-fPIC,-ffp-contract=off",
        *[os.path.join(_HERE, s) for s in _SOURCES],
        "-o", LIB_PATH + ".tmp", "-lpthread",
    ]


def build_popen():
    """Start the build; the caller waits on the returned process."""
    return subprocess.Popen(build_command(), stdout=subprocess.PIPE,
                            stderr=subprocess.STDOUT, text=True)


def finish_build(proc):
    out, _ = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError("synth build failed:\n" + out)
    os.replace(LIB_PATH + ".tmp", LIB_PATH)


def build():
    finish_build(build_popen())


_lib = None

_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
_D = ctypes.c_double
_P = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        common = [_U64, _U32, _U64, _U64, _D, _I64, _D, _D]
        for name in ("syn_fill_f32", "syn_fill_bf16"):
            f = getattr(L, name)
            f.argtypes = [_P, _I64, _I64, *common, ctypes.c_int]
            f.restype = ctypes.c_int
        for name in ("syn_at_f32", "syn_at_bf16"):
            f = getattr(L, name)
            f.argtypes = [_P, _P, _I64, *common, ctypes.c_int]
            f.restype = ctypes.c_int
        for name in ("syn_fill_f32_dev", "syn_fill_bf16_dev"):
            f = getattr(L, name)
            f.argtypes = [_P, _I64, _I64, *common, _P]
            f.restype = ctypes.c_int
        L.syn_log_host.argtypes = [_D]
        L.syn_log_host.restype = _D
        L.syn_key_host.argtypes = [_U64] * 5
        L.syn_key_host.restype = _U64
        L.syn_threshold_host.argtypes = [_D]
        L.syn_threshold_host.restype = _U64
        _lib = L
    return _lib


def _threads(threads):
    if threads is None:
        return max(1, min(os.cpu_count() or 1, 64))
    return threads


def _common(seed, stream, step, rank, sigma, p_limit, outlier_frac, outlier_scale):
    return (seed, stream, step, rank, float(sigma), int(p_limit), float(outlier_frac),
            float(outlier_scale))


def fill(n, *, index0=0, seed=0, stream=STREAM_GRAD, step=0, rank=0, sigma=1e-3,
         p_limit=None, outlier_frac=0.0, outlier_scale=1.0, bf16=False, threads=None):
    """Host fill of ``n`` values at global indices ``index0 .. index0+n-1``.

    Returns float32, or uint16 bf16 bit patterns when ``bf16``.
    """
    p_limit = index0 + n if p_limit is None else p_limit
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    f = lib().syn_fill_bf16 if bf16 else lib().syn_fill_f32
    rc = f(out.ctypes.data, n, index0,
           *_common(seed, stream, step, rank, sigma, p_limit, outlier_frac, outlier_scale),
           _threads(threads))
    if rc != 0:
        raise ValueError("syn_fill failed")
    return out


def at(indices, *, seed=0, stream=STREAM_GRAD, step=0, rank=0, sigma=1e-3, p_limit,
       outlier_frac=0.0, outlier_scale=1.0, bf16=False, threads=None):
    """Host values at arbitrary global indices (for sampled checks)."""
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    out = np.empty(idx.size, dtype=np.uint16 if bf16 else np.float32)
    f = lib().syn_at_bf16 if bf16 else lib().syn_at_f32
    rc = f(out.ctypes.data, idx.ctypes.data, idx.size,
           *_common(seed, stream, step, rank, sigma, p_limit, outlier_frac, outlier_scale),
           _threads(threads))
    if rc != 0:
        raise ValueError("syn_at failed")
    return out


def fill_device(ptr, n, *, index0=0, seed=0, stream=STREAM_GRAD, step=0, rank=0,
                sigma=1e-3, p_limit=None, outlier_frac=0.0, outlier_scale=1.0,
                bf16=False, cuda_stream=0):
    """Device fill of ``n`` values into the device buffer at ``ptr`` (async)."""
    p_limit = index0 + n if p_limit is None else p_limit
    f = lib().syn_fill_bf16_dev if bf16 else lib().syn_fill_f32_dev
    rc = f(ptr, n, index0,
           *_common(seed, stream, step, rank, sigma, p_limit, outlier_frac, outlier_scale),
           cuda_stream)
    if rc != 0:
        raise RuntimeError(f"syn device fill failed ({rc})")
