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


def test_range_casts_are_the_pinned_element_casts(orc):
    """The bf16 and 3-byte range casts the GPU exhaustive test compares with."""
    import pins
    pins.pin_cast_ranges(orc)
