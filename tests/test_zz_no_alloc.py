"""The norm pass for callers that cannot allocate device memory.

Some users of this library cannot hand it scratch memory: a plug-in whose host
application owns the device's memory through an allocator the plug-in cannot
reach, or a training job that has run out of device memory and still needs the
gradient norm to decide whether to skip the step or to log why a rank failed.
zs_grad_sqnorm_noalloc serves them from a static device array inside the
library. This file checks, through the C ABI, that two calls in a row each give
the value the regular entry point (caller-owned scratch) gives for the same
input, within the tolerance the other norm tests use. It is named to be
collected last and sets up everything it needs itself, so it also passes when
run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _slices(plan, seed, bf16, front=0):
    out = []
    for j in range(plan.world):
        h = synth.fill(plan.S, seed=seed, rank=j, step=1, bf16=bf16, outlier_frac=0.01,
                       outlier_scale=100.0)
        buf = torch.zeros(h.nbytes + 64, dtype=torch.uint8, device=DEV)
        view = buf.narrow(0, front, h.nbytes)
        view.copy_(torch.from_numpy(h.view(np.uint8)).to(DEV))
        out.append(view)
    return out


def _regular(plan, lo, hi, slices, gdt):
    ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    zs.zs_grad_sqnorm(plan, 0, lo, hi, slices, gdt, ws, out)
    torch.cuda.synchronize()
    return float(out.item())


def _noalloc(plan, lo, hi, slices, gdt):
    out = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
    zs.zs_grad_sqnorm_noalloc(plan, 0, lo, hi, slices, gdt, out)
    torch.cuda.synchronize()
    return float(out.item())


def _close(a, b, n):
    # The tolerance of the other norm tests: a sequential double sum's bound.
    return abs(a - b) <= (n + 16) * 2.0 ** -52 * abs(b)


def test_two_calls_in_a_row_match_the_regular_entry_point():
    cases = [
        (8, 1 << 20, True, 0, 0, 1 << 20),            # 32-byte aligned: vector path
        (4, 300_000, False, 16, 777, 299_123),        # fp32 slices, 16-byte aligned, ragged range
    ]
    for N, S, bf16, front, lo, hi in cases:
        plan = zs.zs_flatten_plan([N * S], world=N, align_elems=1)
        gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
        first = _slices(plan, 11, bf16, front)
        second = _slices(plan, 12, bf16, front)
        ref1 = _regular(plan, lo, hi, first, gdt)
        ref2 = _regular(plan, lo, hi, second, gdt)
        got1 = _noalloc(plan, lo, hi, first, gdt)
        got2 = _noalloc(plan, lo, hi, second, gdt)
        assert ref1 > 0 and ref2 > 0 and ref1 != ref2
        assert _close(got1, ref1, hi - lo), (got1, ref1)
        assert _close(got2, ref2, hi - lo), (got2, ref2)
        plan.free()
