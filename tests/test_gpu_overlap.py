"""Launch overlap (programmatic dependent launch, zs_set_launch_overlap): the
library's kernels may be scheduled while the previous kernel in the stream
drains, and each waits for its predecessors before touching global memory.
Chains of dependent calls back to back on one stream must give the same bits
with the overlap on and off, and the oracle's bits: steps on the same state in
a row, bucket after bucket, accumulation into the step, the norm pass into
the coefficient into the clipped step, the step into the gather that copies
its slot, a row copy-out after it."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import DEV, assert_state_close, oracle_hp

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _chain(overlap):
    """One stream, no synchronisation between calls; returns host copies."""
    old = zs.zs_set_launch_overlap(overlap)
    try:
        N, S = 4, 3 * (1 << 20) + 4096
        plan = zs.zs_flatten_plan([N * S - 777], world=N, align_elems=128)
        S = plan.S
        stream = torch.cuda.current_stream().cuda_stream
        grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
        master = torch.empty(S, dtype=torch.float32, device=DEV)
        synth.fill_device(master.data_ptr(), S, seed=3, stream=synth.STREAM_MASTER, sigma=0.02,
                          bf16=False, cuda_stream=stream)
        m = torch.zeros(S, dtype=torch.float32, device=DEV)
        v = torch.zeros(S, dtype=torch.float32, device=DEV)
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        other = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        acc = torch.empty(S, dtype=torch.float32, device=DEV)
        ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)
        parts = torch.zeros(N, dtype=torch.float64, device=DEV)
        coef = torch.zeros(1, dtype=torch.float32, device=DEV)
        bad = torch.zeros(1, dtype=torch.int32, device=DEV)
        cut = S // 3 + 5
        for t in range(1, 4):
            for j, g in enumerate(grads):
                synth.fill_device(g.data_ptr(), S, seed=3, rank=j, step=t, sigma=1e-3, bf16=True,
                                  cuda_stream=stream)
            # two bucket calls, then the same state again at once
            zs.zs_shard_step(plan, 1, 0, cut, grads, zs.ZS_BF16, master, m, v, full, zs.ZS_BF16,
                             HP, 2 * t - 1)
            zs.zs_shard_step(plan, 1, cut, S, grads, zs.ZS_BF16, master, m, v, full, zs.ZS_BF16,
                             HP, 2 * t - 1)
            zs.zs_grad_accumulate(plan, 1, 0, S, grads, zs.ZS_BF16, acc, True)
            for r in range(N):
                zs.zs_grad_sqnorm(plan, 1, 0, S, grads, zs.ZS_BF16, ws, parts.narrow(0, r, 1))
            zs.zs_clip_coefficient(parts, N, 0.01, coef, bad)
            zs.zs_shard_step_accumulated_clipped(plan, 1, 0, S, grads, zs.ZS_BF16, acc, 2, master,
                                                 m, v, full, zs.ZS_BF16, HP, 2 * t, coef, bad)
            # the gather reads the slot the step just wrote
            srcs = [None] * N
            srcs[1] = full.narrow(0, S, S)
            zs.zs_gather_assemble(plan, 0, srcs, other, zs.ZS_BF16)
        torch.cuda.synchronize()
        zs.zs_check_device_error()
        out = [x.cpu().numpy().view(np.uint32) for x in (master, m, v)]
        out += [full.cpu().numpy().view(np.uint16), other.cpu().numpy().view(np.uint16),
                coef.cpu().numpy().view(np.uint32), parts.cpu().numpy().view(np.uint64)]
        plan.free()
        return out
    finally:
        zs.zs_set_launch_overlap(old)


def test_overlap_on_and_off_give_the_same_bits():
    on, off = _chain(1), _chain(0)
    for k, (a, b) in enumerate(zip(on, off)):
        assert np.array_equal(a, b), k
    # the gather copied exactly the slot the last step wrote
    S = on[0].size
    assert np.array_equal(on[4][S:2 * S], on[3][S:2 * S])


def test_back_to_back_steps_match_the_oracle(orc):
    """Ten steps on the same state in a row with nothing between the launches
    (each must wait for the previous one's writes), against the oracle."""
    assert zs.zs_set_launch_overlap(1) in (0, 1)
    N, S = 8, (1 << 21) + 512
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
    g_host = [synth.fill(S, seed=9, rank=j, step=1, bf16=True) for j in range(N)]
    master0 = synth.fill(S, seed=9, stream=synth.STREAM_MASTER, sigma=0.02)
    d_g = [torch.from_numpy(x.view(np.int16)).to(DEV) for x in g_host]
    d = [torch.from_numpy(master0.copy()).to(DEV), torch.zeros(S, device=DEV),
         torch.zeros(S, device=DEV)]
    full = torch.zeros(N * S, dtype=torch.int16, device=DEV)
    o = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(N * S, np.uint16)
    for t in range(1, 11):
        zs.zs_shard_step(plan, 0, 0, S, d_g, zs.ZS_BF16, *d, full, zs.ZS_BF16, HP, t)
        orc.shard_step(world=N, rank=0, S=S, lo=0, hi=S, grads=g_host, master=o[0], m=o[1],
                       v=o[2], full_flat=o_full, t=t, **oracle_hp(HP))
    torch.cuda.synchronize()
    for name, x, ref in zip(("master", "m", "v"), d, o):
        assert assert_state_close(x.cpu().numpy(), ref, name) == 0
    assert np.array_equal(full.cpu().numpy().view(np.uint16), o_full)
    plan.free()


def test_overlap_switch_rejects_other_values():
    with pytest.raises(ValueError):
        zs.zs_set_launch_overlap(2)
