"""CPU oracle for the ZeRO/FSDP shard-local step — TEST INFRASTRUCTURE.

A plain, slow, single-threaded C++ restatement (``oracle.cpp``) of what the
shard-local step computes, with numpy-facing wrappers. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
may import this package. It shares no code with the CUDA path, and the
product library never calls it.

Build: ``g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared`` (no fast-math),
so each float operation is one IEEE binary32 op rounded to nearest even.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "oracle.cpp")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

BF16, FP32, FP24 = 0, 1, 2
ELEM_BYTES = {BF16: 2, FP32: 4, FP24: 3}
STAGE_DDP, STAGE_ZERO1, STAGE_ZERO2, STAGE_ZERO3 = 0, 1, 2, 3

CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build_command(src=SRC, out=LIB_PATH + ".tmp", extra=()):
    return ["g++", *CXXFLAGS, *extra, src, "-o", out]


def build_popen():
    return subprocess.Popen(build_command(), stdout=subprocess.PIPE,
                            stderr=subprocess.STDOUT, text=True)


def finish_build(proc):
    out, _ = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + out)
    os.replace(LIB_PATH + ".tmp", LIB_PATH)


def build():
    finish_build(build_popen())


_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_D = ctypes.c_double
_F = ctypes.c_float
_P = ctypes.c_void_p


def load(path=LIB_PATH):
    """Load an oracle library (the default one, or a test's variant build)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    L.oracle_plan.argtypes = [_P, _P, _I32, _I32, _I64, _I64, _P, _P, _P, _P, _I32]
    L.oracle_plan.restype = ctypes.c_int
    L.oracle_shard_range.argtypes = [_I64, _I64, _I32, _I64, _P, _P]
    L.oracle_shard_range.restype = None
    L.oracle_ledger_bytes_per_param.argtypes = [_I32, _I32]
    L.oracle_ledger_bytes_per_param.restype = _D
    L.oracle_ledger_kept_bytes.argtypes = [_I32, _I64, _I32]
    L.oracle_ledger_kept_bytes.restype = _I64
    L.oracle_adamw_scalars.argtypes = [_D, _D, _D, _D, _D, _I64, _I32, _P]
    L.oracle_adamw_scalars.restype = None
    L.oracle_shard_step.argtypes = [_I32, _I32, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P,
                                    _I32, _D, _D, _D, _D, _D, _I64]
    L.oracle_shard_step.restype = ctypes.c_int
    L.oracle_ddp_step.argtypes = [_I32, _I64, _P, _I32, _P, _P, _P, _P, _I32, _D, _D, _D,
                                  _D, _D, _I64]
    L.oracle_ddp_step.restype = ctypes.c_int
    L.oracle_grad_sqnorm.argtypes = [_I32, _I64, _I64, _I64, _P, _I32]
    L.oracle_grad_sqnorm.restype = _D
    L.oracle_clip_coef.argtypes = [_P, _I32, _D, _P, _P]
    L.oracle_clip_coef.restype = None
    L.oracle_shard_step_clipped.argtypes = [_I32, _I32, _I64, _I64, _I64, _P, _I32, _P, _P, _P,
                                            _P, _I32, _D, _D, _D, _D, _D, _I64, _F, _I32]
    L.oracle_shard_step_clipped.restype = ctypes.c_int
    L.oracle_grad_accumulate.argtypes = [_I32, _I64, _I64, _I64, _P, _I32, _P, _I32]
    L.oracle_grad_accumulate.restype = ctypes.c_int
    L.oracle_shard_step_accumulated.argtypes = [_I32, _I32, _I64, _I64, _I64, _P, _I32, _P, _I32,
                                                _P, _P, _P, _P, _I32, _D, _D, _D, _D, _D, _I64]
    L.oracle_shard_step_accumulated.restype = ctypes.c_int
    L.oracle_grad_sqnorm_accumulated.argtypes = [_I32, _I64, _I64, _I64, _P, _I32, _P, _I32]
    L.oracle_grad_sqnorm_accumulated.restype = _D
    L.oracle_shard_step_accumulated_clipped.argtypes = [_I32, _I32, _I64, _I64, _I64, _P, _I32,
                                                        _P, _I32, _P, _P, _P, _P, _I32, _D, _D,
                                                        _D, _D, _D, _I64, _F, _I32]
    L.oracle_shard_step_accumulated_clipped.restype = ctypes.c_int
    L.oracle_rows_plan.argtypes = [_P, _P, _P, _I32, _I32, _I64, _P, _P, _P, _P]
    L.oracle_rows_plan.restype = ctypes.c_int
    L.oracle_unshard.argtypes = [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _P, _P]
    L.oracle_unshard.restype = None
    L.oracle_shard_rows.argtypes = [_P, _P, _P, _P, _P, _I32, _I32, _I64, _I32, _P, _P]
    L.oracle_shard_rows.restype = None
    L.oracle_gather.argtypes = [_I32, _I64, _I32, _P, _P]
    L.oracle_gather.restype = None
    L.oracle_bf16_rne.argtypes = [_F]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_fp24_rne.argtypes = [_F]
    L.oracle_fp24_rne.restype = ctypes.c_uint32
    L.oracle_bf16_rne_array.argtypes = [_P, _P, _I64]
    L.oracle_bf16_rne_array.restype = None
    L.oracle_bf16_rne_bits_range.argtypes = [ctypes.c_uint32, _I64, _P]
    L.oracle_bf16_rne_bits_range.restype = None
    L.oracle_fp24_rne_bits_range.argtypes = [ctypes.c_uint32, _I64, _P]
    L.oracle_fp24_rne_bits_range.restype = None
    return L


class Oracle:
    """numpy-facing wrappers over one loaded oracle library."""

    def __init__(self, path=LIB_PATH):
        self.L = load(path)

    # -- O1 plan ---------------------------------------------------------
    def plan(self, numels, tied_to=None, world=1, align=128, bucket_elems=0):
        numels = np.ascontiguousarray(numels, dtype=np.int64)
        n = numels.size
        tied = None if tied_to is None else np.ascontiguousarray(tied_to, dtype=np.int32)
        offsets = np.zeros(max(n, 1), dtype=np.int64)
        info = np.zeros(4, dtype=np.int64)
        cap = max(n, 1) + 1
        blo = np.zeros(cap, dtype=np.int64)
        bhi = np.zeros(cap, dtype=np.int64)
        rc = self.L.oracle_plan(numels.ctypes.data if n else None,
                                tied.ctypes.data if tied is not None else None, n, world,
                                align, bucket_elems, offsets.ctypes.data, info.ctypes.data,
                                blo.ctypes.data, bhi.ctypes.data, cap)
        if rc != 0:
            raise ValueError(f"oracle_plan rejected the input ({rc})")
        nb = int(info[3])
        return dict(P=int(info[0]), P_pad=int(info[1]), S=int(info[2]),
                    offsets=offsets[:n].copy(),
                    buckets=[(int(blo[b]), int(bhi[b])) for b in range(nb)])

    def shard_range(self, flo, fhi, rank, S):
        lo = ctypes.c_int64()
        hi = ctypes.c_int64()
        self.L.oracle_shard_range(flo, fhi, rank, S, ctypes.byref(lo), ctypes.byref(hi))
        return lo.value, hi.value

    # -- O2 ledger -------------------------------------------------------
    def ledger_bytes_per_param(self, stage, world):
        return self.L.oracle_ledger_bytes_per_param(stage, world)

    def ledger_kept_bytes(self, stage, P_pad, world):
        return self.L.oracle_ledger_kept_bytes(stage, P_pad, world)

    # -- O3-O5 step ------------------------------------------------------
    def scalars(self, lr, beta1, beta2, eps, wd, t, world):
        out = np.zeros(10, dtype=np.float32)
        self.L.oracle_adamw_scalars(lr, beta1, beta2, eps, wd, t, world, out.ctypes.data)
        return out

    @staticmethod
    def _ptrs(arrays):
        return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data if a is not None else None
                                                 for a in arrays])

    def shard_step(self, *, world, rank, S, lo, hi, grads, master, m, v, full_flat,
                   param_dtype=BF16, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01,
                   t=1):
        """In place on master/m/v (float32 [S]) and full_flat (param bytes)."""
        g0 = grads[0]
        gdt = BF16 if g0.dtype == np.uint16 else FP32
        for g in grads:
            assert g.dtype == g0.dtype and g.size >= S and g.flags.c_contiguous
        for a in (master, m, v):
            assert a.dtype == np.float32 and a.size >= S and a.flags.c_contiguous
        assert len(grads) == world
        rc = self.L.oracle_shard_step(world, rank, S, lo, hi, self._ptrs(grads), gdt,
                                      master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                      full_flat.ctypes.data, param_dtype, lr, beta1, beta2,
                                      eps, wd, t)
        if rc != 0:
            raise ValueError("oracle_shard_step rejected the input")

    def ddp_step(self, *, world, P_pad, local_grads, master, m, v, params,
                 param_dtype=BF16, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01, t=1):
        gdt = BF16 if local_grads[0].dtype == np.uint16 else FP32
        rc = self.L.oracle_ddp_step(world, P_pad, self._ptrs(local_grads), gdt,
                                    master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                    params.ctypes.data, param_dtype, lr, beta1, beta2, eps,
                                    wd, t)
        if rc != 0:
            raise ValueError("oracle_ddp_step rejected the input")

    # -- global-norm clipping ---------------------------------------------
    def grad_sqnorm(self, *, world, S, lo, hi, grads):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        return self.L.oracle_grad_sqnorm(world, S, lo, hi, self._ptrs(grads), gdt)

    def clip_coef(self, rank_sqnorms, max_norm):
        a = np.ascontiguousarray(rank_sqnorms, dtype=np.float64)
        coef = ctypes.c_float()
        bad = ctypes.c_int32()
        self.L.oracle_clip_coef(a.ctypes.data, a.size, max_norm, ctypes.byref(coef),
                                ctypes.byref(bad))
        return np.float32(coef.value), int(bad.value)

    def shard_step_clipped(self, *, world, rank, S, lo, hi, grads, master, m, v, full_flat,
                           coef, skip, param_dtype=BF16, lr=1e-3, beta1=0.9, beta2=0.999,
                           eps=1e-8, wd=0.01, t=1):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        rc = self.L.oracle_shard_step_clipped(world, rank, S, lo, hi, self._ptrs(grads), gdt,
                                              master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                              full_flat.ctypes.data, param_dtype, lr, beta1,
                                              beta2, eps, wd, t, float(coef), int(skip))
        if rc != 0:
            raise ValueError("oracle_shard_step_clipped rejected the input")

    # -- gradient accumulation ------------------------------------------
    def grad_accumulate(self, *, world, S, lo, hi, grads, accum, first):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        assert accum.dtype == np.float32 and accum.size >= S
        rc = self.L.oracle_grad_accumulate(world, S, lo, hi, self._ptrs(grads), gdt,
                                           accum.ctypes.data, 1 if first else 0)
        if rc != 0:
            raise ValueError("oracle_grad_accumulate rejected the input")

    def shard_step_accumulated(self, *, world, rank, S, lo, hi, grads, accum, micro_steps,
                               master, m, v, full_flat, param_dtype=BF16, lr=1e-3, beta1=0.9,
                               beta2=0.999, eps=1e-8, wd=0.01, t=1):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        rc = self.L.oracle_shard_step_accumulated(world, rank, S, lo, hi, self._ptrs(grads), gdt,
                                                  accum.ctypes.data, micro_steps,
                                                  master.ctypes.data, m.ctypes.data,
                                                  v.ctypes.data, full_flat.ctypes.data,
                                                  param_dtype, lr, beta1, beta2, eps, wd, t)
        if rc != 0:
            raise ValueError("oracle_shard_step_accumulated rejected the input")

    # -- clipping an accumulated gradient ---------------------------------
    def grad_sqnorm_accumulated(self, *, world, S, lo, hi, grads, accum, micro_steps):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        assert accum.dtype == np.float32 and accum.size >= S
        return self.L.oracle_grad_sqnorm_accumulated(world, S, lo, hi, self._ptrs(grads), gdt,
                                                     accum.ctypes.data, micro_steps)

    def shard_step_accumulated_clipped(self, *, world, rank, S, lo, hi, grads, accum,
                                       micro_steps, master, m, v, full_flat, coef, skip,
                                       param_dtype=BF16, lr=1e-3, beta1=0.9, beta2=0.999,
                                       eps=1e-8, wd=0.01, t=1):
        gdt = BF16 if grads[0].dtype == np.uint16 else FP32
        rc = self.L.oracle_shard_step_accumulated_clipped(
            world, rank, S, lo, hi, self._ptrs(grads), gdt, accum.ctypes.data, micro_steps,
            master.ctypes.data, m.ctypes.data, v.ctypes.data, full_flat.ctypes.data, param_dtype,
            lr, beta1, beta2, eps, wd, t, float(coef), int(skip))
        if rc != 0:
            raise ValueError("oracle_shard_step_accumulated_clipped rejected the input")

    # -- per-parameter row sharding (FSDP2) ------------------------------
    def rows_plan(self, dim0, numels, tied_to=None, world=1, align=128):
        n = len(numels)
        d = np.ascontiguousarray(dim0, dtype=np.int64)
        ne = np.ascontiguousarray(numels, dtype=np.int64)
        tied = None if tied_to is None else np.ascontiguousarray(tied_to, dtype=np.int32)
        off = np.zeros(max(n, 1), np.int64)
        c = np.zeros(max(n, 1), np.int64)
        w = np.zeros(max(n, 1), np.int64)
        S = ctypes.c_int64()
        rc = self.L.oracle_rows_plan(d.ctypes.data, ne.ctypes.data,
                                     tied.ctypes.data if tied is not None else None, n, world,
                                     align, off.ctypes.data, c.ctypes.data, w.ctypes.data,
                                     ctypes.byref(S))
        if rc != 0:
            raise ValueError("oracle_rows_plan rejected the input")
        return dict(S=S.value, offsets=off[:n].copy(), rows_per_rank=c[:n].copy(),
                    row_elems=w[:n].copy(), dim0=d, tied=tied, world=world, n=n)

    def unshard(self, rp, gathered, elem_size, params):
        self.L.oracle_unshard(rp["dim0"].ctypes.data, rp["offsets"].ctypes.data,
                              rp["rows_per_rank"].ctypes.data, rp["row_elems"].ctypes.data,
                              rp["tied"].ctypes.data if rp["tied"] is not None else None, rp["n"],
                              rp["world"], rp["S"], elem_size, gathered.ctypes.data,
                              self._ptrs(params))

    def shard_rows(self, rp, rank, elem_size, params, local):
        self.L.oracle_shard_rows(rp["dim0"].ctypes.data, rp["offsets"].ctypes.data,
                                 rp["rows_per_rank"].ctypes.data, rp["row_elems"].ctypes.data,
                                 rp["tied"].ctypes.data if rp["tied"] is not None else None,
                                 rp["n"], rank, rp["S"], elem_size, self._ptrs(params),
                                 local.ctypes.data)

    # -- sharded checkpoint: what a restore must produce ------------------
    # "从 Data Parallel 到 ZeRO/FSDP", "Checkpoint 不能假设每个 Rank 都有完整模型":
    # each rank's shard is a piece of global tensors that the metadata
    # describes; a restore into another world size (or layout) is the same
    # global tensors cut the new way. Written here as exactly that: gather the
    # global tensors from all old shards, then cut the new rank's shard.
    # A layout is ("flat", numels, tied, world, align) or ("rows", rows_plan dict).
    def global_params(self, layout, shards):
        """The fp32 tensors of every owner parameter from all ranks' shards
        (None for tied entries)."""
        if layout[0] == "flat":
            _, numels, tied, world, align = layout
            pl = self.plan(numels, tied, world=world, align=align)
            flat = np.concatenate([np.ascontiguousarray(s[:pl["S"]]) for s in shards])
            return [None if (tied is not None and tied[i] >= 0) else
                    flat[pl["offsets"][i]:pl["offsets"][i] + numels[i]].copy()
                    for i in range(len(numels))]
        rp = layout[1]
        gathered = np.concatenate([np.ascontiguousarray(s[:rp["S"]]) for s in shards])
        params = [None if (rp["tied"] is not None and rp["tied"][i] >= 0) else
                  np.zeros(int(rp["dim0"][i] * rp["row_elems"][i]), np.float32)
                  for i in range(rp["n"])]
        self.unshard(rp, gathered.view(np.uint8), 4,
                     [None if p is None else p.view(np.uint8) for p in params])
        return params

    def shard_of(self, layout, params, rank):
        """Rank ``rank``'s fp32 shard of the given global tensors (padding 0)."""
        if layout[0] == "flat":
            _, numels, tied, world, align = layout
            pl = self.plan(numels, tied, world=world, align=align)
            flat = np.zeros(pl["P_pad"], np.float32)
            for i, p in enumerate(params):
                if p is not None:
                    flat[pl["offsets"][i]:pl["offsets"][i] + numels[i]] = p
            return flat[rank * pl["S"]:(rank + 1) * pl["S"]].copy()
        rp = layout[1]
        local = np.zeros(rp["S"], np.float32)
        self.shard_rows(rp, rank, 4, [None if p is None else p.view(np.uint8) for p in params],
                        local.view(np.uint8))
        return local

    def reshard(self, old_layout, old_shards, new_layout, rank):
        return self.shard_of(new_layout, self.global_params(old_layout, old_shards), rank)

    # -- O6 gather -------------------------------------------------------
    def gather(self, *, world, S, elem_size, shards, full_flat):
        self.L.oracle_gather(world, S, elem_size, self._ptrs(shards), full_flat.ctypes.data)

    # -- casts -----------------------------------------------------------
    def bf16(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.size, dtype=np.uint16)
        self.L.oracle_bf16_rne_array(x.ctypes.data, out.ctypes.data, x.size)
        return out

    def bf16_bits_range(self, first, n):
        out = np.empty(n, dtype=np.uint16)
        self.L.oracle_bf16_rne_bits_range(first, n, out.ctypes.data)
        return out

    def fp24_bits_range(self, first, n):
        """3 bytes per value (little-endian) of the patterns first .. first+n-1
        (mod 2^32) cast to the 3-byte parameter type."""
        out = np.empty(3 * n, dtype=np.uint8)
        self.L.oracle_fp24_rne_bits_range(first & 0xFFFFFFFF, n, out.ctypes.data)
        return out

    def fp24(self, x):
        return int(self.L.oracle_fp24_rne(float(x)))


_default = None


def default():
    global _default
    if _default is None:
        _default = Oracle()
    return _default
