"""The step's cast of the fp32 master into the parameter slot, on the GPU, over
all 2^32 fp32 bit patterns, against the oracle's casts ("从 Data Parallel 到
ZeRO/FSDP", "Mixed Precision 至少有四个 Dtype": the fp32 master is kept and a
low-precision copy of it is what the ranks gather).

Each chunk of patterns is the master of one step with lr = 0, weight decay 0,
zero gradient slices and eps > 0: then m = v = 0, the update is 0 / eps = 0
and the master is multiplied by fp32(1 - 0) = 1 and has 0 subtracted, which
leaves every non-NaN pattern's bits as they are (no flush of subnormals;
-0 - 0 = -0), so the slot holds the cast of the pattern itself. NaN patterns
must give a NaN (the payload is not specified: the GPU's arithmetic may
replace it before the cast).

Covered: the register-streaming kernel's 32-byte group path (bf16 through
cvt.rn.bf16x2, the 3-byte rounding, the fp32 copy), the staged kernel (bf16
and 3-byte), and the element-by-element path (cvt.rn.bf16 and the 3-byte
rounding one value at a time, taken for a slot that is not vector-aligned:
rank 1 of 2 with an odd shard length)."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
from gpu_util import DEV

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(os.environ.get("ZS_BOUNDS_CHECK") == "1",
                       reason="every pattern runs in the ordinary suite"),
]

HP0 = dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
CHUNK = 1 << 28
ALL = 1 << 32
THREADS = max(1, min(os.cpu_count() or 1, 32))


def _patterns_dev(first, n):
    """fp32 tensor whose element i has the bit pattern (first + i) mod 2^32."""
    x = torch.arange(first, first + n, dtype=torch.int64, device=DEV) % ALL
    x = torch.where(x >= (1 << 31), x - ALL, x)
    return x.to(torch.int32).view(torch.float32)


def _nan_intervals(first, n):
    """Index intervals [a, b) of the chunk whose patterns are NaNs (exponent all
    ones, mantissa non-zero): 0x7F800001..0x7FFFFFFF and 0xFF800001..0xFFFFFFFF,
    also where the chunk wraps past 2^32."""
    out = []
    for base in (0, ALL):
        for lo, hi in ((0x7F800001, 0x80000000), (0xFF800001, ALL)):
            a, b = max(lo + base, first), min(hi + base, first + n)
            if a < b:
                out.append((a - first, b - first))
    return out


def _expected(orc, first, n, pdt):
    """The oracle's cast of the chunk's patterns, computed on all host cores."""
    eb = oracle.ELEM_BYTES[pdt]
    out = np.empty(n * eb, np.uint8)
    parts = np.linspace(0, n, THREADS + 1).astype(np.int64)

    def work(a, b):
        if pdt == oracle.BF16:
            out[2 * a:2 * b] = orc.bf16_bits_range((first + a) % ALL, b - a).view(np.uint8)
        elif pdt == oracle.FP24:
            out[3 * a:3 * b] = orc.fp24_bits_range((first + a) % ALL, b - a)
        else:  # the fp32 parameter is the master itself
            out[4 * a:4 * b] = (np.arange(first + a, first + b, dtype=np.uint64) % ALL).astype(
                np.uint32).view(np.uint8)

    with cf.ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(work, parts[:-1], parts[1:]))
    return out


def _is_nan(raw, pdt):
    """NaN test on the slot's stored values (uint8 bytes of one interval)."""
    if pdt == oracle.BF16:
        h = raw.view(np.uint16)
        return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)
    if pdt == oracle.FP32:
        w = raw.view(np.uint32)
        return ((w & 0x7F800000) == 0x7F800000) & ((w & 0x007FFFFF) != 0)
    b = raw.reshape(-1, 3).astype(np.uint32)
    q = b[:, 0] | (b[:, 1] << 8) | (b[:, 2] << 16)
    return ((q & 0x7F8000) == 0x7F8000) & ((q & 0x007FFF) != 0)


def _compare(got, want, first, n, pdt, what):
    eb = oracle.ELEM_BYTES[pdt]
    nans = _nan_intervals(first, n)
    for a, b in nans:
        assert _is_nan(got[eb * a:eb * b], pdt).all(), f"{what}: a NaN pattern lost its NaN"
        got[eb * a:eb * b] = want[eb * a:eb * b]
    if np.array_equal(got, want):
        return
    bad = np.nonzero((got.reshape(-1, eb) != want.reshape(-1, eb)).any(axis=1))[0]
    i = int(bad[0])
    raise AssertionError(f"{what}: {bad.size} patterns differ, first 0x{(first + i) % ALL:08x}: "
                         f"got {got[eb * i:eb * i + eb].tolist()} want "
                         f"{want[eb * i:eb * i + eb].tolist()}")


class _Runner:
    """Device buffers for one plan, reused across chunks."""

    def __init__(self, world, rank, S, align):
        self.plan = zs.zs_flatten_plan([world * S], world=world, align_elems=align)
        assert self.plan.S == S
        self.world, self.rank, self.S = world, rank, S
        self.slices = [torch.zeros(S, dtype=torch.int16, device=DEV) for _ in range(world)]
        self.m = torch.empty(S, dtype=torch.float32, device=DEV)
        self.v = torch.empty(S, dtype=torch.float32, device=DEV)
        self.full = torch.empty(world * S * 4, dtype=torch.uint8, device=DEV)

    def slot(self, master, pdt, zdt, path):
        eb = oracle.ELEM_BYTES[pdt]
        self.m.zero_()
        self.v.zero_()
        old = zs.zs_set_step_path(path)
        try:
            zs.zs_shard_step(self.plan, self.rank, 0, self.S, self.slices, zs.ZS_BF16, master,
                             self.m, self.v, self.full, zdt, HP0, 1)
            kernel = zs.zs_last_step_kernel()
        finally:
            zs.zs_set_step_path(old)
        off = self.rank * self.S * eb
        got = self.full[off:off + self.S * eb].cpu().numpy()
        return got, kernel

    def free(self):
        self.plan.free()


ZDT = {oracle.BF16: zs.ZS_BF16, oracle.FP24: zs.ZS_FP24, oracle.FP32: zs.ZS_FP32}


def test_cast_all_patterns_vector_paths(orc):
    """2^32 patterns in 16 chunks of 2^28: the register-streaming kernel's
    32-byte groups (bf16, 3-byte, fp32 parameters) and the staged kernel's
    tiles (bf16, 3-byte); the master comes back unchanged (NaN as NaN)."""
    run = _Runner(world=1, rank=0, S=CHUNK, align=128)
    cases = [(oracle.BF16, zs.STEP_PATH_DIRECT, (1, 16)), (oracle.FP24, zs.STEP_PATH_DIRECT, (1, 16)),
             (oracle.FP32, zs.STEP_PATH_DIRECT, (1, 16)), (oracle.BF16, zs.STEP_PATH_STAGED, (2, None)),
             (oracle.FP24, zs.STEP_PATH_STAGED, (2, None))]
    for first in range(0, ALL, CHUNK):
        master = _patterns_dev(first, CHUNK)
        want = {p: _expected(orc, first, CHUNK, p) for p in (oracle.BF16, oracle.FP24, oracle.FP32)}
        for pdt, path, kernel in cases:
            got, k = run.slot(master, pdt, ZDT[pdt], path)
            assert k[0] == kernel[0] and (kernel[1] is None or k[1] == kernel[1]), k
            _compare(got, want[pdt], first, CHUNK, pdt, f"path {path} dtype {pdt}")
        # p * 1 - 0 kept every pattern (the master is fp32, no flush to zero)
        back = master.view(torch.int32).cpu().numpy().view(np.uint8)
        _compare(back, want[oracle.FP32], first, CHUNK, oracle.FP32, "master")
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    run.free()


def test_cast_all_patterns_element_path(orc):
    """2^32 patterns (16 chunks of 2^28 + 1, the last wrapping to pattern 0)
    through the element-by-element path: rank 1 of 2 with an odd shard length,
    so the slot is not aligned for vector stores; bf16 and 3-byte parameters."""
    S = CHUNK + 1
    run = _Runner(world=2, rank=1, S=S, align=1)
    for first in range(0, ALL, S):
        master = _patterns_dev(first, S)
        for pdt in (oracle.BF16, oracle.FP24):
            want = _expected(orc, first, S, pdt)
            got, k = run.slot(master, pdt, ZDT[pdt], zs.STEP_PATH_DIRECT)
            assert k == (1, 0), k
            _compare(got, want, first, S, pdt, f"element path dtype {pdt}")
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    run.free()
