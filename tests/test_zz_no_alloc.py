"""The norm pass for callers that cannot allocate device memory.

Some users of this library cannot hand it scratch memory: a plug-in whose host
application owns the device's memory through an allocator the plug-in cannot
reach, or a training job that has run out of device memory and still needs the
gradient norm to decide whether to skip the step or to log why a rank failed.
zs_grad_sqnorm_noalloc serves them from a static device array inside the
library. This file checks, through the C ABI, that two calls in a row each give
exactly the value the regular entry point (caller-owned scratch) gives for the
same input, that both agree with the oracle's sum within the tolerance the
other norm tests use, and that the calls allocate no device memory. It is
named to be collected last and sets up everything it needs itself, so it also
passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _slices(host, front=0):
    out = []
    for h in host:
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


def _bits(x):
    return int(np.array([x], dtype=np.float64).view(np.uint64)[0])


def _sum_bound(n):
    # The tolerance of the other norm tests: a sequential double sum's bound.
    return (n + 16) * 2.0 ** -52


def test_two_calls_in_a_row_match_the_regular_entry_point():
    """Both entry points launch the same deterministic norm pass (same kernel,
    same grid, same fixed-order reduction); only where the scratch lives
    differs. So each no-alloc call must give exactly the regular call's bits,
    and both must be within a sequential sum's rounding bound of the oracle's
    sum. The two calls in a row see different inputs, so a partial or ticket
    left over from the first call would show in the second. Around the two
    calls nothing is allocated on the device: free device memory and the
    caching allocator's allocation count stay as they were."""
    orc = oracle.default()
    cases = [
        (8, 1 << 20, True, 0, 0, 1 << 20),            # 32-byte aligned: vector path
        (4, 300_000, False, 16, 777, 299_123),        # fp32 slices, 16-byte aligned, ragged range
    ]
    for N, S, bf16, front, lo, hi in cases:
        plan = zs.zs_flatten_plan([N * S], world=N, align_elems=1)
        gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
        host = {seed: [synth.fill(plan.S, seed=seed, rank=j, step=1, bf16=bf16,
                                  outlier_frac=0.01, outlier_scale=100.0) for j in range(N)]
                for seed in (11, 12)}
        first = _slices(host[11], front)
        second = _slices(host[12], front)
        ref1 = _regular(plan, lo, hi, first, gdt)
        ref2 = _regular(plan, lo, hi, second, gdt)
        outs = [torch.full((1,), -1.0, dtype=torch.float64, device=DEV) for _ in range(3)]
        # One call first: the library looks its array up on this device, and
        # the kernel's module is loaded; then the two calls measured.
        zs.zs_grad_sqnorm_noalloc(plan, 0, lo, hi, second, gdt, outs[0])
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        zs.zs_grad_sqnorm_noalloc(plan, 0, lo, hi, first, gdt, outs[1])
        zs.zs_grad_sqnorm_noalloc(plan, 0, lo, hi, second, gdt, outs[2])
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
        assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
        got1, got2 = float(outs[1].item()), float(outs[2].item())
        assert ref1 > 0 and ref2 > 0 and ref1 != ref2
        assert _bits(got1) == _bits(ref1), (got1, ref1)
        assert _bits(got2) == _bits(ref2), (got2, ref2)
        for got, seed in ((got1, 11), (got2, 12)):
            want = orc.grad_sqnorm(world=N, S=plan.S, lo=lo, hi=hi, grads=host[seed])
            assert abs(got - want) <= _sum_bound(hi - lo) * want, (got, want)
        plan.free()
