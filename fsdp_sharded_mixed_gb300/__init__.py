"""GB300-native shard-local step for ZeRO-1/2/3 and FSDP.

A thin ctypes binding over ``libzs.so`` (the C ABI in ``include/zs.h``): the
functions here carry the C names and only marshal arguments — tensor data
pointers, sizes, the CUDA stream handle — to the library, whose CUDA kernels
do every step of the path. PyTorch supplies device memory and streams. There
is no fallback: without the compiled library every call raises.

Entry points: ``zs_flatten_plan`` (flat layout, rank shards, buckets),
``zs_shard_step`` (N-slice fp32 mean + AdamW + cast into the AllGather slot),
``zs_gather_assemble`` (the AllGather's result and per-tensor views); the
FSDP2 row layout (``zs_rows_plan``, ``zs_unshard``, ``zs_shard_rows``);
clipping, accumulation, and the sharded checkpoint (``zs_checkpoint_save``,
``zs_checkpoint_load``: host file I/O of host- or device-resident state).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
CSRC = os.path.join(_HERE, "csrc")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_HERE, "libzs.so")
# The same library with every kernel access checked against its launch's
# window (CUDA sources compiled with ZS_BOUNDS_CHECK=1); loaded instead of
# libzs.so when the environment variable ZS_BOUNDS_CHECK is 1.
CHECKED_LIB_PATH = os.path.join(_HERE, "libzs_checked.so")
INCLUDE = os.path.join(_ROOT, "include")

ZS_OK, ZS_ERR_INVAL, ZS_ERR_ALIGN, ZS_ERR_RANGE = 0, -1, -2, -3
ZS_ERR_CUDA, ZS_ERR_NOMEM, ZS_ERR_TIMEOUT, ZS_ERR_UNSUPPORTED = -4, -5, -6, -7
ZS_ERR_IO, ZS_ERR_CORRUPT = -8, -9
ZS_BF16, ZS_FP32, ZS_FP24 = 0, 1, 2
ELEM_BYTES = {ZS_BF16: 2, ZS_FP32: 4, ZS_FP24: 3}
ZS_MAX_WORLD = 1024

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-fmad=false", "-prec-div=true",
              "-prec-sqrt=true", "-ftz=false", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-pthread", "-I/usr/local/cuda/include"]
CUDA_SOURCES = ["shard_step.cu", "gather.cu", "clip.cu", "accum.cu", "rows.cu", "ckpt.cu"]
HOST_SOURCES = ["api.cpp", "plan.cpp", "checkpoint.cpp", "trace.cpp"]


# ----------------------------------------------------------------- build ----
def _compile_jobs():
    """(command, object, variant) per translation unit: the CUDA sources once
    per variant ("" ordinary, "checked" bounds-checked), the host sources once
    (they are the same in both libraries)."""
    jobs = []
    for variant, defs in (("", []), ("checked", ["-DZS_BOUNDS_CHECK=1"])):
        for src in CUDA_SOURCES:
            obj = os.path.join(BUILD_DIR, variant, src + ".o")
            jobs.append((["nvcc", "-c", *NVCC_FLAGS, *defs, os.path.join(CSRC, src), "-o", obj],
                         obj, variant))
    for src in HOST_SOURCES:
        obj = os.path.join(BUILD_DIR, src + ".o")
        jobs.append((["g++", "-c", *CXX_FLAGS, os.path.join(CSRC, src), "-o", obj], obj, None))
    return jobs


def build(log=True):
    """Compile both libraries for sm_103a in-tree (sources in parallel) and
    link them: libzs.so and the bounds-checked libzs_checked.so."""
    os.makedirs(os.path.join(BUILD_DIR, "checked"), exist_ok=True)
    jobs = _compile_jobs()

    def run(job):
        cmd = job[0]
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p.returncode, p.stdout + p.stderr

    with ThreadPoolExecutor(len(jobs)) as ex:
        results = list(ex.map(run, jobs))
    report = []
    for cmd, rc, out in results:
        report.append("$ " + " ".join(cmd) + "\n" + out)
        if rc != 0:
            raise RuntimeError("libzs build failed:\n" + out)
    for variant, path in (("", LIB_PATH), ("checked", CHECKED_LIB_PATH)):
        objs = [o for _, o, v in jobs if v in (variant, None)]
        link = ["nvcc", "-shared", *ARCH, "-o", path + ".tmp", *objs]
        p = subprocess.run(link, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"{os.path.basename(path)} link failed:\n" + p.stdout + p.stderr)
        os.replace(path + ".tmp", path)
    if log:
        with open(os.path.join(BUILD_DIR, "build.log"), "w") as f:
            f.write("\n".join(report))


# ------------------------------------------------------------------- ABI ----
class ZsError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


_lib = None
_I32, _I64, _P = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p


class AdamWHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double)]


EXPORTS = {
    "zs_flatten_plan": ([_P, _P, _I32, _I32, _I64, _I64, _P], ctypes.c_int),
    "zs_plan_info": ([_P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "zs_plan_offsets": ([_P, _P, _I32], ctypes.c_int),
    "zs_plan_bucket_range": ([_P, _I32, _P, _P], ctypes.c_int),
    "zs_plan_bucket": ([_P, _I32, _I32, _P, _P], ctypes.c_int),
    "zs_plan_free": ([_P], ctypes.c_int),
    "zs_shard_step": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _P, _P, _P, ctypes.c_int,
                       ctypes.POINTER(AdamWHparams), _I64, _P], ctypes.c_int),
    "zs_shard_step_to_shard": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _P, _P, _P,
                                ctypes.c_int, ctypes.POINTER(AdamWHparams), _I64, _P],
                               ctypes.c_int),
    "zs_gather_assemble": ([_P, _I32, _P, _P, ctypes.c_int, _P, _P], ctypes.c_int),
    "zs_grad_norm_workspace_bytes": ([], _I64),
    "zs_grad_sqnorm": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _I64, _P, _P], ctypes.c_int),
    "zs_grad_sqnorm_noalloc": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _P], ctypes.c_int),
    "zs_clip_coefficient": ([_P, _I32, ctypes.c_double, _P, _P, _P], ctypes.c_int),
    "zs_shard_step_clipped": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _P, _P, _P,
                               ctypes.c_int, ctypes.POINTER(AdamWHparams), _I64, _P, _P, _P],
                              ctypes.c_int),
    "zs_grad_accumulate": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _I32, _P], ctypes.c_int),
    "zs_shard_step_accumulated": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _I32, _P, _P, _P,
                                   _P, ctypes.c_int, ctypes.POINTER(AdamWHparams), _I64, _P],
                                  ctypes.c_int),
    "zs_grad_sqnorm_accumulated": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _I32, _P, _I64,
                                    _P, _P], ctypes.c_int),
    "zs_shard_step_accumulated_clipped": ([_P, _I32, _I64, _I64, _P, ctypes.c_int, _P, _I32, _P,
                                           _P, _P, _P, ctypes.c_int,
                                           ctypes.POINTER(AdamWHparams), _I64, _P, _P, _P],
                                          ctypes.c_int),
    "zs_rows_plan": ([_P, _P, _P, _I32, _I32, _I64, _P], ctypes.c_int),
    "zs_plan_rows": ([_P, _P, _P, _I32], ctypes.c_int),
    "zs_unshard": ([_P, _P, ctypes.c_int, _P, _P], ctypes.c_int),
    "zs_shard_rows": ([_P, _I32, _P, ctypes.c_int, _P, _P], ctypes.c_int),
    "zs_checkpoint_save": ([_P, _I32, _P, _P, _P, _I64, ctypes.c_char_p, _P], ctypes.c_int),
    "zs_checkpoint_load": ([_P, _I32, _P, _I32, _P, _P, _P, _P, _P], ctypes.c_int),
    "zs_checkpoint_info": ([ctypes.c_char_p, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "zs_checkpoint_release_staging": ([], ctypes.c_int),
    "zs_set_trace": ([ctypes.c_char_p], ctypes.c_int),
    "zs_trace_first_divergence": ([_P, _I32, _P, ctypes.c_char_p, _I64], ctypes.c_int),
    "zs_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "zs_last_error": ([], ctypes.c_char_p),
    "zs_check_device_error": ([_P], ctypes.c_int),
    "zs_set_validation": ([_I32], _I32),
    "zs_set_step_path": ([_I32], _I32),
    "zs_last_step_kernel": ([_P, _P], ctypes.c_int),
    "zs_set_launch_overlap": ([_I32], _I32),
    "zs_selftest_wait_timeout": ([ctypes.c_uint32, _P], ctypes.c_int),
    "zs_bounds_checked": ([], _I32),
    "zs_selftest_bounds_window": ([_I64], ctypes.c_int),
    "zs_version": ([], ctypes.c_char_p),
}


def lib_path():
    """The library this process uses: libzs_checked.so when ZS_BOUNDS_CHECK=1."""
    return CHECKED_LIB_PATH if os.environ.get("ZS_BOUNDS_CHECK") == "1" else LIB_PATH


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: the CUDA library must be built "
                               "(__graft_entry__.build()); there is no fallback")
        L = ctypes.CDLL(path)
        for name, (args, res) in EXPORTS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(status):
    if status != ZS_OK:
        L = lib()
        detail = L.zs_last_error().decode() or L.zs_status_string(status).decode()
        raise ZsError(status, detail)


def _ptr(x):
    """Address of a tensor or a numpy array (or an int address / None). The
    library reads and writes buffers as dense runs of bytes, so a strided
    view is refused rather than passed by its first element's address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("zs: tensor arguments must be contiguous")
        return x.data_ptr()
    if not x.flags["C_CONTIGUOUS"]:
        raise ValueError("zs: array arguments must be C-contiguous")
    return x.ctypes.data


class Buffers:
    """A list of buffers (the N gradient slices, say) marshalled once: their
    addresses in a ready C array, each checked dense, and the smallest byte
    size among them. Pass it wherever a list of slices goes to skip the
    per-call work (about half a microsecond per buffer) in calls repeated with
    the same buffers, e.g. ReduceScatter outputs reused every step."""

    def __init__(self, bufs):
        bufs = list(bufs)
        self.array = (ctypes.c_void_p * max(len(bufs), 1))(*[_ptr(b) for b in bufs])
        sizes = [x.nbytes for x in bufs if x is not None and not isinstance(x, int)]
        self.min_nbytes = min(sizes) if len(sizes) == len(bufs) and sizes else None
        self._n = len(bufs)

    def __len__(self):
        return self._n


def _slices(bufs):
    """The C array of a slice list's addresses."""
    if isinstance(bufs, Buffers):
        return bufs.array
    return (ctypes.c_void_p * max(len(bufs), 1))(*[_ptr(g) for g in bufs])


def _need(x, nbytes, fn, name, index=None):
    """A tensor or array argument must hold the bytes the call touches (raw
    addresses are the caller's responsibility; the library checks device
    allocations where the driver can tell)."""
    if x is None or isinstance(x, int):
        return
    have = x.nbytes  # torch.Tensor and numpy.ndarray alike
    if have < nbytes:
        label = name if index is None else f"{name}[{index}]"
        raise ValueError(f"{fn}: {label} holds {have} bytes, the call needs {nbytes}")


def _step_sizes(fn, plan, lo, hi, grad_slices, grad_dtype, states, out, param_dtype,
                out_elems, accum=None):
    """The byte sizes the step family needs: N slices of S gradient elements,
    fp32 [S] states (and accumulator), the output of out_elems parameters."""
    if hi <= lo:
        return
    S = plan.S
    gbytes = S * ELEM_BYTES[grad_dtype]
    if isinstance(grad_slices, Buffers):
        if grad_slices.min_nbytes is not None and grad_slices.min_nbytes < gbytes:
            raise ValueError(f"{fn}: a gradient slice holds {grad_slices.min_nbytes} bytes, "
                             f"the call needs {gbytes}")
    else:
        for j, g in enumerate(grad_slices):
            _need(g, gbytes, fn, "grad_slices", j)
    for name, x in zip(("master", "exp_avg", "exp_avg_sq"), states):
        _need(x, S * 4, fn, name)
    if out is not None:
        _need(out, out_elems * ELEM_BYTES.get(param_dtype, 0), fn, "output")
    if accum is not None:
        _need(accum, S * 4, fn, "accum")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a ``zs_plan*``; freed when garbage-collected or by ``free()``."""

    def __init__(self, handle, n_params, rows=False):
        self.handle = handle
        self.n_params = n_params
        self.rows = rows  # made by zs_rows_plan (per-parameter row sharding)
        info = zs_plan_info(self)
        self.P, self.P_pad, self.S = info["P"], info["P_pad"], info["S"]
        self.n_buckets, self.world = info["n_buckets"], info["world"]

    def free(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check(lib().zs_plan_free(h))

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def zs_flatten_plan(numels, tied_to=None, world=1, align_elems=128, bucket_elems=0):
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*numels)
    ties = None if tied_to is None else (ctypes.c_int32 * max(n, 1))(*tied_to)
    out = ctypes.c_void_p()
    _check(lib().zs_flatten_plan(arr, ties, n, world, align_elems, bucket_elems,
                                 ctypes.byref(out)))
    return Plan(out.value, n)


def zs_rows_plan(dim0, numels, tied_to=None, world=1, align_elems=128):
    """Per-parameter row sharding (FSDP2 Shard(0)); see include/zs.h."""
    n = len(numels)
    d = (ctypes.c_int64 * max(n, 1))(*dim0)
    arr = (ctypes.c_int64 * max(n, 1))(*numels)
    ties = None if tied_to is None else (ctypes.c_int32 * max(n, 1))(*tied_to)
    out = ctypes.c_void_p()
    _check(lib().zs_rows_plan(d, arr, ties, n, world, align_elems, ctypes.byref(out)))
    return Plan(out.value, n, rows=True)


def zs_plan_rows(plan):
    c = (ctypes.c_int64 * max(plan.n_params, 1))()
    w = (ctypes.c_int64 * max(plan.n_params, 1))()
    _check(lib().zs_plan_rows(plan.handle, c, w, plan.n_params))
    return list(c)[:plan.n_params], list(w)[:plan.n_params]


def zs_unshard(plan, gathered, dtype, params_out, stream=None):
    ptrs = (ctypes.c_void_p * max(len(params_out), 1))(*[_ptr(p) for p in params_out])
    _check(lib().zs_unshard(plan.handle, _ptr(gathered), dtype, ptrs, _stream(stream)))


def zs_shard_rows(plan, rank, params_in, dtype, local_out, stream=None):
    ptrs = (ctypes.c_void_p * max(len(params_in), 1))(*[_ptr(p) for p in params_in])
    _check(lib().zs_shard_rows(plan.handle, rank, ptrs, dtype, _ptr(local_out), _stream(stream)))


def zs_plan_info(plan):
    P, P_pad, S = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    nb, w, npar = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(lib().zs_plan_info(plan.handle, ctypes.byref(P), ctypes.byref(P_pad),
                              ctypes.byref(S), ctypes.byref(nb), ctypes.byref(w),
                              ctypes.byref(npar)))
    return dict(P=P.value, P_pad=P_pad.value, S=S.value, n_buckets=nb.value, world=w.value,
                n_params=npar.value)


def zs_plan_offsets(plan):
    out = (ctypes.c_int64 * max(plan.n_params, 1))()
    _check(lib().zs_plan_offsets(plan.handle, out, plan.n_params))
    return list(out)[:plan.n_params]


def zs_plan_bucket_range(plan, bucket):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zs_plan_bucket_range(plan.handle, bucket, ctypes.byref(lo), ctypes.byref(hi)))
    return lo.value, hi.value


def zs_plan_bucket(plan, bucket, rank):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zs_plan_bucket(plan.handle, bucket, rank, ctypes.byref(lo), ctypes.byref(hi)))
    return lo.value, hi.value


def zs_shard_step(plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg, exp_avg_sq,
                  full_flat, param_dtype, hp, step, stream=None):
    """Enqueue rank ``rank``'s fused step over shard-local ``[lo, hi)``.

    ``grad_slices``: N device tensors (or addresses); ``master``/``exp_avg``/
    ``exp_avg_sq``: fp32 [S]; ``full_flat``: N*S elements of ``param_dtype``;
    ``hp``: dict with lr, beta1, beta2, eps, weight_decay; ``step`` >= 1.
    """
    _step_sizes("zs_shard_step", plan, lo, hi, grad_slices, grad_dtype,
                (master, exp_avg, exp_avg_sq), full_flat, param_dtype, plan.P_pad)
    ptrs = _slices(grad_slices)
    h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    _check(lib().zs_shard_step(plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(master),
                               _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(full_flat), param_dtype,
                               ctypes.byref(h), step, _stream(stream)))


def zs_shard_step_to_shard(plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg,
                           exp_avg_sq, param_shard, param_dtype, hp, step, stream=None):
    """``zs_shard_step`` writing the cast parameters into ``param_shard`` (S
    elements of ``param_dtype``) instead of the rank's slot of the flat buffer."""
    _step_sizes("zs_shard_step_to_shard", plan, lo, hi, grad_slices, grad_dtype,
                (master, exp_avg, exp_avg_sq), param_shard, param_dtype, plan.S)
    ptrs = _slices(grad_slices)
    h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    _check(lib().zs_shard_step_to_shard(plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(master),
                                        _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(param_shard),
                                        param_dtype, ctypes.byref(h), step, _stream(stream)))


def zs_shard_step_clipped(plan, rank, lo, hi, grad_slices, grad_dtype, master, exp_avg,
                          exp_avg_sq, full_flat, param_dtype, hp, step, coef=None, skip=None,
                          stream=None):
    """``zs_shard_step`` with a device clip coefficient and skip flag (tensors
    or addresses of a device fp32 and a device int32; None = not used)."""
    _step_sizes("zs_shard_step_clipped", plan, lo, hi, grad_slices, grad_dtype,
                (master, exp_avg, exp_avg_sq), full_flat, param_dtype, plan.P_pad)
    ptrs = _slices(grad_slices)
    h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    _check(lib().zs_shard_step_clipped(plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(master),
                                       _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(full_flat),
                                       param_dtype, ctypes.byref(h), step, _ptr(coef),
                                       _ptr(skip), _stream(stream)))


def zs_grad_accumulate(plan, rank, lo, hi, grad_slices, grad_dtype, accum, first, stream=None):
    """Enqueue accum = (first ? 0 : accum) + mean of the slices (fp32 [S])."""
    _step_sizes("zs_grad_accumulate", plan, lo, hi, grad_slices, grad_dtype, (), None, 0, 0,
                accum)
    ptrs = _slices(grad_slices)
    _check(lib().zs_grad_accumulate(plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(accum),
                                    1 if first else 0, _stream(stream)))


def zs_shard_step_accumulated(plan, rank, lo, hi, grad_slices, grad_dtype, accum, micro_steps,
                              master, exp_avg, exp_avg_sq, full_flat, param_dtype, hp, step,
                              stream=None):
    """The step on ((accum + mean of the slices) / micro_steps)."""
    _step_sizes("zs_shard_step_accumulated", plan, lo, hi, grad_slices, grad_dtype,
                (master, exp_avg, exp_avg_sq), full_flat, param_dtype, plan.P_pad, accum)
    ptrs = _slices(grad_slices)
    h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    _check(lib().zs_shard_step_accumulated(plan.handle, rank, lo, hi, ptrs, grad_dtype,
                                           _ptr(accum), micro_steps, _ptr(master),
                                           _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(full_flat),
                                           param_dtype, ctypes.byref(h), step, _stream(stream)))


def zs_grad_sqnorm_accumulated(plan, rank, lo, hi, grad_slices, grad_dtype, accum, micro_steps,
                               workspace, sqnorm_out, stream=None):
    """Enqueue the shard's sum of squares of the accumulated step's gradient
    ((accum + mean) * (1/G)) into the device double ``sqnorm_out``."""
    _step_sizes("zs_grad_sqnorm_accumulated", plan, lo, hi, grad_slices, grad_dtype, (), None,
                0, 0, accum)
    ptrs = _slices(grad_slices)
    nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") \
        else zs_grad_norm_workspace_bytes()
    _check(lib().zs_grad_sqnorm_accumulated(plan.handle, rank, lo, hi, ptrs, grad_dtype,
                                            _ptr(accum), micro_steps, _ptr(workspace), nbytes,
                                            _ptr(sqnorm_out), _stream(stream)))


def zs_shard_step_accumulated_clipped(plan, rank, lo, hi, grad_slices, grad_dtype, accum,
                                      micro_steps, master, exp_avg, exp_avg_sq, full_flat,
                                      param_dtype, hp, step, coef=None, skip=None, stream=None):
    """The accumulated step with a device clip coefficient and skip flag."""
    _step_sizes("zs_shard_step_accumulated_clipped", plan, lo, hi, grad_slices, grad_dtype,
                (master, exp_avg, exp_avg_sq), full_flat, param_dtype, plan.P_pad, accum)
    ptrs = _slices(grad_slices)
    h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"])
    _check(lib().zs_shard_step_accumulated_clipped(
        plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(accum), micro_steps, _ptr(master),
        _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(full_flat), param_dtype, ctypes.byref(h), step,
        _ptr(coef), _ptr(skip), _stream(stream)))


def zs_grad_norm_workspace_bytes():
    return lib().zs_grad_norm_workspace_bytes()


def zs_grad_sqnorm(plan, rank, lo, hi, grad_slices, grad_dtype, workspace, sqnorm_out,
                   stream=None):
    """Enqueue the shard's sum of squared mean gradients into the device
    double ``sqnorm_out``; ``workspace`` is caller-owned device scratch."""
    _step_sizes("zs_grad_sqnorm", plan, lo, hi, grad_slices, grad_dtype, (), None, 0, 0)
    ptrs = _slices(grad_slices)
    nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") \
        else zs_grad_norm_workspace_bytes()
    _check(lib().zs_grad_sqnorm(plan.handle, rank, lo, hi, ptrs, grad_dtype, _ptr(workspace),
                                nbytes, _ptr(sqnorm_out), _stream(stream)))


def zs_grad_sqnorm_noalloc(plan, rank, lo, hi, grad_slices, grad_dtype, sqnorm_out,
                           stream=None):
    """``zs_grad_sqnorm`` for callers that cannot allocate device memory: the
    scratch is the library's own static device array (see include/zs.h for
    the first-call set-up and for why overlapping calls must not be issued)."""
    _step_sizes("zs_grad_sqnorm_noalloc", plan, lo, hi, grad_slices, grad_dtype, (), None, 0, 0)
    ptrs = _slices(grad_slices)
    _check(lib().zs_grad_sqnorm_noalloc(plan.handle, rank, lo, hi, ptrs, grad_dtype,
                                        _ptr(sqnorm_out), _stream(stream)))


def zs_clip_coefficient(rank_sqnorms, n, max_norm, coef_out, nonfinite_out, stream=None):
    _check(lib().zs_clip_coefficient(_ptr(rank_sqnorms), n, max_norm, _ptr(coef_out),
                                     _ptr(nonfinite_out), _stream(stream)))


def zs_gather_assemble(plan, rank, shard_srcs, full_flat, param_dtype, stream=None):
    """Enqueue the assembly of the other ranks' shards into ``full_flat``;
    return the per-parameter device addresses (the unflattened views)."""
    eb = ELEM_BYTES.get(param_dtype, 0)
    if isinstance(shard_srcs, Buffers):
        if shard_srcs.min_nbytes is not None and shard_srcs.min_nbytes < plan.S * eb:
            raise ValueError(f"zs_gather_assemble: a shard holds {shard_srcs.min_nbytes} "
                             f"bytes, the call needs {plan.S * eb}")
    else:
        for j, x in enumerate(shard_srcs):
            _need(x, plan.S * eb, "zs_gather_assemble", "shard_srcs", j)
    _need(full_flat, plan.P_pad * eb, "zs_gather_assemble", "full_flat")
    srcs = _slices(shard_srcs)
    views = None if plan.rows else (ctypes.c_void_p * max(plan.n_params, 1))()
    _check(lib().zs_gather_assemble(plan.handle, rank, srcs, _ptr(full_flat), param_dtype,
                                    views, _stream(stream)))
    if views is None:  # row-sharded: the buffer is rank-major; see zs_unshard
        return None
    return [v or 0 for v in list(views)[:plan.n_params]]


def _io_stream(stream):
    """The stream for a checkpoint call: as given, else the current CUDA
    stream where there is a device, else NULL (host-resident state)."""
    if stream is not None:
        return _stream(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None


def zs_checkpoint_save(plan, rank, master, exp_avg, exp_avg_sq, step, path, stream=None):
    """Write rank ``rank``'s fp32 master/exp_avg/exp_avg_sq shard (S elements
    each; device tensors, or host tensors / numpy arrays) and the global step
    to ``path``. Blocks until the file is complete."""
    for name, x in zip(("master", "exp_avg", "exp_avg_sq"), (master, exp_avg, exp_avg_sq)):
        _need(x, plan.S * 4, "zs_checkpoint_save", name)
    _check(lib().zs_checkpoint_save(plan.handle, rank, _ptr(master), _ptr(exp_avg),
                                    _ptr(exp_avg_sq), step, os.fsencode(path),
                                    _io_stream(stream)))


def zs_checkpoint_load(plan, rank, paths, master, exp_avg, exp_avg_sq, stream=None):
    """Fill rank ``rank``'s shard of ``plan`` from the files of the old ranks
    (``paths[k]`` = old rank k's file; None for a file this rank does not
    need, never for rank 0); returns the saved step."""
    for name, x in zip(("master", "exp_avg", "exp_avg_sq"), (master, exp_avg, exp_avg_sq)):
        _need(x, plan.S * 4, "zs_checkpoint_load", name)
    arr = (ctypes.c_char_p * max(len(paths), 1))(
        *[None if p is None else os.fsencode(p) for p in paths])
    step = ctypes.c_int64()
    _check(lib().zs_checkpoint_load(plan.handle, rank, arr, len(paths), _ptr(master),
                                    _ptr(exp_avg), _ptr(exp_avg_sq), ctypes.byref(step),
                                    _io_stream(stream)))
    return step.value


def zs_checkpoint_release_staging():
    """Free the pinned staging kept between checkpoint calls."""
    _check(lib().zs_checkpoint_release_staging())


def zs_checkpoint_info(path):
    w, r, lay, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    P, S, step = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zs_checkpoint_info(os.fsencode(path), ctypes.byref(w), ctypes.byref(r),
                                    ctypes.byref(lay), ctypes.byref(n), ctypes.byref(P),
                                    ctypes.byref(S), ctypes.byref(step)))
    return dict(world=w.value, rank=r.value, layout=lay.value, n_params=n.value, P=P.value,
                S=S.value, step=step.value)


def zs_selftest_wait_timeout(polls, stream=None):
    """Enqueue a bounded wait that runs out (see include/zs.h)."""
    _check(lib().zs_selftest_wait_timeout(polls, _stream(stream)))


def zs_bounds_checked():
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().zs_bounds_checked())


def zs_selftest_bounds_window(shrink):
    """Bounds-checked build only: narrow the window the step, accumulation and
    norm kernels check against by ``shrink`` elements at each end (0 = off)."""
    _check(lib().zs_selftest_bounds_window(shrink))


def zs_set_trace(path):
    """Per-call trace to ``path`` (``%r`` = RANK, ``%p`` = pid); None = off."""
    _check(lib().zs_set_trace(None if path is None else os.fsencode(path)))


def zs_trace_first_divergence(paths):
    """The first record at which the ranks' traces disagree: (index, detail),
    or None when they agree throughout."""
    arr = (ctypes.c_char_p * len(paths))(*[os.fsencode(p) for p in paths])
    seq = ctypes.c_int64()
    buf = ctypes.create_string_buffer(8192)
    _check(lib().zs_trace_first_divergence(arr, len(paths), ctypes.byref(seq), buf, len(buf)))
    return None if seq.value < 0 else (seq.value, buf.value.decode())


def zs_check_device_error(stream=None):
    _check(lib().zs_check_device_error(_stream(stream)))


def zs_set_validation(level):
    return lib().zs_set_validation(level)


STEP_PATH_AUTO, STEP_PATH_DIRECT, STEP_PATH_STAGED = 0, 1, 2


def zs_set_step_path(path):
    """0 = kernel chosen per call, 1 = register-streaming, 2 = staged (bulk
    async copies into shared memory) where it applies; returns the old path."""
    old = lib().zs_set_step_path(path)
    if old < 0:
        raise ValueError(f"unknown step path {path}")
    return old


def zs_set_launch_overlap(on):
    """1: launches may overlap the previous kernel's drain (programmatic
    dependent launch; results unchanged), 0: ordinary launches. Returns the
    previous setting."""
    old = lib().zs_set_launch_overlap(int(on))
    if old < 0:
        raise ValueError(f"launch overlap must be 0 or 1, got {on}")
    return old


def zs_last_step_kernel():
    """(kernel, elems) of the calling thread's last step-family launch: (1, 16 /
    8 / 0) register-streaming with that vector group, (2, 2048 / 1024) staged
    with that tile; (0, 0) before the first."""
    k, e = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().zs_last_step_kernel(ctypes.byref(k), ctypes.byref(e)))
    return k.value, e.value


def zs_version():
    return lib().zs_version().decode()


def tensor_views(full_flat, addresses, shapes):
    """Wrap the addresses ``zs_gather_assemble`` returned as views of the
    ``full_flat`` tensor with the given shapes (no copy)."""
    base = full_flat.data_ptr()
    es = full_flat.element_size()
    out = []
    for addr, shape in zip(addresses, shapes):
        off = (addr - base) // es
        n = 1
        for d in shape:
            n *= d
        out.append(full_flat.narrow(0, off, n).view(shape))
    return out
