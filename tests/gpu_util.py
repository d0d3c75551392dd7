"""Helpers for the GPU parity tests: device buffers from the seeded generator,
and the comparison gates (fp32 state: max relative error 1e-6, NaN matches
NaN; low-precision parameters: at most 1 ulp; layout: bit-exact)."""
from __future__ import annotations

import numpy as np
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle as orc
import synth

REL_TOL = 1e-6
DEV = torch.device("cuda:0")

ZS_OF = {orc.BF16: zs.ZS_BF16, orc.FP32: zs.ZS_FP32, orc.FP24: zs.ZS_FP24}


def to_dev(a):
    """numpy array -> device tensor with the same bytes."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV)
    if a.dtype == np.uint8:
        return torch.from_numpy(a).to(DEV)
    return torch.from_numpy(a).to(DEV)


def to_host(t, dtype):
    return t.cpu().numpy().view(dtype)


def dev_fill(n, *, bf16, **kw):
    t = torch.empty(n, dtype=torch.int16 if bf16 else torch.float32, device=DEV)
    synth.fill_device(t.data_ptr(), n, bf16=bf16,
                      cuda_stream=torch.cuda.current_stream().cuda_stream, **kw)
    return t


def all_zero(t, chunk=1 << 28):
    """True when every element of the device tensor is zero; checked a chunk at
    a time so that no temporary the size of a large buffer is allocated."""
    flat = t.reshape(-1)
    for i in range(0, flat.numel(), chunk):
        if bool(flat[i:i + chunk].any()):
            return False
    return True


def assert_state_close(got, ref, name):
    """fp32 gate: max |a-b|/max(|a|,|b|) <= 1e-6 (0/0 = 0), NaN only with NaN."""
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{name}: NaN pattern differs"
    a, b = got[~gn].astype(np.float64), ref[~rn].astype(np.float64)
    inf = np.isinf(a) | np.isinf(b)
    assert np.array_equal(a[inf], b[inf]), f"{name}: infinities differ"
    a, b = a[~inf], b[~inf]
    den = np.maximum(np.abs(a), np.abs(b))
    rel = np.where(den > 0, np.abs(a - b) / np.where(den > 0, den, 1), 0.0)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= REL_TOL, f"{name}: max relative error {worst:.3g} > {REL_TOL}"
    return int(np.count_nonzero(got.view(np.uint32) != ref.view(np.uint32)))


def _ordered(bits, width):
    """Map sign-magnitude float patterns of `width` bits to ordered integers."""
    b = bits.astype(np.int64)
    sign = 1 << (width - 1)
    return np.where(b & sign, -(b & (sign - 1)), b)


def assert_params_close(got_bytes, ref_bytes, param_dtype, name="params"):
    """Low-precision parameter gate: at most 1 ulp apart, NaN with NaN."""
    if param_dtype == orc.FP32:
        return assert_state_close(got_bytes.view(np.float32), ref_bytes.view(np.float32), name)
    if param_dtype == orc.BF16:
        g, r, width, exp_mask, man_mask = got_bytes.view(np.uint16), ref_bytes.view(np.uint16), \
            16, 0x7F80, 0x007F
    else:
        gb = got_bytes.reshape(-1, 3).astype(np.int64)
        rb = ref_bytes.reshape(-1, 3).astype(np.int64)
        g = gb[:, 0] | (gb[:, 1] << 8) | (gb[:, 2] << 16)
        r = rb[:, 0] | (rb[:, 1] << 8) | (rb[:, 2] << 16)
        width, exp_mask, man_mask = 24, 0x7F8000, 0x007FFF
    g = np.asarray(g, np.int64)
    r = np.asarray(r, np.int64)
    gnan = ((g & exp_mask) == exp_mask) & ((g & man_mask) != 0)
    rnan = ((r & exp_mask) == exp_mask) & ((r & man_mask) != 0)
    assert np.array_equal(gnan, rnan), f"{name}: NaN pattern differs"
    d = np.abs(_ordered(g[~gnan], width) - _ordered(r[~rnan], width))
    worst = int(d.max()) if d.size else 0
    assert worst <= 1, f"{name}: {worst} ulp apart"
    return int(np.count_nonzero(g[~gnan] != r[~rnan]))


def oracle_hp(hp):
    return dict(lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                wd=hp["weight_decay"])
