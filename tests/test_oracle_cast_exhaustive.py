"""The oracle's fp32 -> bf16 rounding against PyTorch's CPU conversion (a
library routine that rounds to nearest even) over all 2^32 fp32 patterns.
NaNs are compared as "both NaN" (PyTorch drops the sign of a NaN)."""
import numpy as np
import torch


def test_bf16_all_patterns(orc):
    chunk = 1 << 24
    for first in range(0, 1 << 32, chunk):
        bits = np.arange(first, first + chunk, dtype=np.uint32)
        ref = torch.from_numpy(bits.view(np.float32)).to(torch.bfloat16).view(torch.int16)
        ref = ref.numpy().view(np.uint16)
        got = orc.bf16_bits_range(first, chunk)
        if np.array_equal(got, ref):
            continue
        bad = np.nonzero(got != ref)[0]
        nan_ref = ((ref[bad] & 0x7F80) == 0x7F80) & ((ref[bad] & 0x7F) != 0)
        nan_got = ((got[bad] & 0x7F80) == 0x7F80) & ((got[bad] & 0x7F) != 0)
        assert np.all(nan_ref & nan_got), \
            f"first mismatch at pattern {hex(int(bits[bad[~(nan_ref & nan_got)][0]]))}"


def test_fp24_range_packs_the_pinned_scalar_cast(orc):
    """The 3-byte range cast (the GPU exhaustive test's expected bytes) is the
    scalar 3-byte rounding pinned against the exact nearest value, stored
    little-endian, over windows around every boundary of the format and a
    window that wraps past 0xFFFFFFFF."""
    starts = [0, 0x7F - 40, 0x00800000 - 300, 0x7F7FFF00 - 200, 0x7F800000 - 300,
              0x7FFFFFFF - 100, 0x80000000 - 20, 0xFF7FFF00, 0xFFFFFFFF - 150]
    rng = np.random.default_rng(5)
    starts += [int(x) for x in rng.integers(0, 1 << 32, size=20)]
    for first in starts:
        n = 700
        got = orc.fp24_bits_range(first, n).reshape(n, 3).astype(np.uint32)
        packed = got[:, 0] | (got[:, 1] << 8) | (got[:, 2] << 16)
        for i in range(0, n, 7):
            bits = (first + i) & 0xFFFFFFFF
            x = np.array([bits], dtype=np.uint32).view(np.float32)[0]
            assert int(packed[i]) == orc.fp24(x), hex(bits)
