"""GPU parity at the edges of the input space, against the oracle, bit for bit,
with guard bands around every output: the largest world the ABI takes
(N = 1024 slices, the kernels' largest parameter blocks) through the step, the
norm pass, the accumulation and the gather; N = 1 (the mean is the slice
itself); one-element shards, one of them all padding; an empty range; and the
staged kernel with N = 16 bf16 slices at exactly the smallest range it takes
(8 whole 2048-element tiles) and one element or one tile short of it."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import DEV, assert_params_close, assert_state_close, oracle_hp, to_dev, to_host

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
CANARY = 0x5A


def guarded(host):
    """(whole, inner): the bytes of ``host`` on the device between 256-byte
    guard bands of CANARY."""
    raw = np.ascontiguousarray(host).view(np.uint8)
    whole = torch.full((raw.size + 512,), CANARY, dtype=torch.uint8, device=DEV)
    inner = whole.narrow(0, 256, raw.size)
    if raw.size:
        inner.copy_(torch.from_numpy(raw).to(DEV))
    return whole, inner


def intact(whole):
    n = whole.numel()
    return bool((whole[:256] == CANARY).all()) and bool((whole[n - 256:] == CANARY).all())


def _step_case(orc, plan, rank, lo, hi, steps=2, seed=0, path=zs.STEP_PATH_AUTO):
    """Run `steps` steps of rank `rank` over [lo, hi) on the GPU and in the
    oracle from the same inputs; compare state, the flat buffer and guards."""
    N, S, P, P_pad = plan.world, plan.S, plan.P, plan.P_pad
    master0 = synth.fill(S, index0=rank * S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02,
                         p_limit=P)
    o_st = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(P_pad, np.uint16)
    d_st = [guarded(x) for x in o_st]
    d_full = guarded(o_full)
    old = zs.zs_set_step_path(path)
    try:
        for t in range(1, steps + 1):
            g = [synth.fill(S, index0=rank * S, seed=seed, rank=j, step=t, p_limit=P, bf16=True)
                 for j in range(N)]
            d_g = [guarded(x) for x in g]
            zs.zs_shard_step(plan, rank, lo, hi, [x[1] for x in d_g], zs.ZS_BF16,
                             *[x[1] for x in d_st], d_full[1], zs.ZS_BF16, HP, t)
            orc.shard_step(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=g, master=o_st[0],
                           m=o_st[1], v=o_st[2], full_flat=o_full, t=t, **oracle_hp(HP))
            zs.zs_check_device_error()
            assert all(intact(x[0]) for x in d_g)
    finally:
        zs.zs_set_step_path(old)
    for name, (whole, inner), ref in zip(("master", "m", "v"), d_st, o_st):
        got = to_host(inner, np.float32)
        assert assert_state_close(got, ref, name) == 0
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), name
        assert intact(whole), name
    got = to_host(d_full[1], np.uint16)
    assert assert_params_close(got.view(np.uint8), o_full.view(np.uint8), oracle.BF16) == 0
    assert np.array_equal(got, o_full) and intact(d_full[0])


def test_max_world_step(orc):
    """N = 1024 (ZS_MAX_WORLD): the last rank, which also holds the padding."""
    plan = zs.zs_flatten_plan([1024 * 97 + 5, 333], world=zs.ZS_MAX_WORLD, align_elems=1)
    assert plan.world == 1024 and plan.P_pad > plan.P
    _step_case(orc, plan, 1023, 0, plan.S, seed=21)
    _step_case(orc, plan, 517, 3, plan.S - 2, seed=22)
    plan.free()


def test_max_world_norm_accumulate_gather(orc):
    N = zs.ZS_MAX_WORLD
    plan = zs.zs_flatten_plan([N * 150], world=N, align_elems=1)
    S = plan.S
    host = [synth.fill(S, seed=23, rank=j, step=1, bf16=True, outlier_frac=0.02,
                       outlier_scale=30.0) for j in range(N)]
    dev = [to_dev(h) for h in host]
    # norm
    ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    zs.zs_grad_sqnorm(plan, 7, 0, S, dev, zs.ZS_BF16, ws, out)
    ref = orc.grad_sqnorm(world=N, S=S, lo=0, hi=S, grads=host)
    assert abs(float(out.item()) - ref) <= (S + 16) * 2.0 ** -52 * ref
    # accumulation, two micro-steps
    acc_w, acc = guarded(np.full(S, np.nan, np.float32))
    o_acc = np.zeros(S, np.float32)
    for k in range(2):
        zs.zs_grad_accumulate(plan, 7, 1, S - 1, dev, zs.ZS_BF16, acc, k == 0)
        orc.grad_accumulate(world=N, S=S, lo=1, hi=S - 1, grads=host, accum=o_acc, first=k == 0)
    got = to_host(acc, np.float32)
    assert np.array_equal(got[1:S - 1].view(np.uint32), o_acc[1:S - 1].view(np.uint32))
    assert np.isnan(got[0]) and np.isnan(got[S - 1]) and intact(acc_w)
    # gather: the other 1023 ranks' shards into their slots; rank 5's own slot
    # already holds its shard (the step wrote it there) and is skipped
    shards = [synth.fill(S, seed=24, rank=j, step=2, bf16=True) for j in range(N)]
    start = np.zeros(plan.P_pad, np.uint16)
    start[5 * S:6 * S] = shards[5]
    full_w, full = guarded(start)
    views = zs.zs_gather_assemble(plan, 5, [to_dev(x) for x in shards], full, zs.ZS_BF16)
    o_full = np.zeros(plan.P_pad, np.uint16)
    orc.gather(world=N, S=S, elem_size=2, shards=shards, full_flat=o_full)
    assert np.array_equal(to_host(full, np.uint16), o_full) and intact(full_w)
    assert views == [full.data_ptr()]
    plan.free()


def test_single_rank(orc):
    """N = 1: the reduce is the slice itself times fp32(1/1) = 1."""
    plan = zs.zs_flatten_plan([777, 5], world=1, align_elems=1)
    assert plan.S == 782
    _step_case(orc, plan, 0, 0, plan.S, steps=3, seed=25)
    _step_case(orc, plan, 0, 13, 700, seed=26)
    plan.free()


def test_one_element_shards(orc):
    one = zs.zs_flatten_plan([1], world=1, align_elems=1)
    assert one.S == 1
    _step_case(orc, one, 0, 0, 1, steps=3, seed=27)
    one.free()
    pad = zs.zs_flatten_plan([3], world=4, align_elems=1)
    assert (pad.P, pad.P_pad, pad.S) == (3, 4, 1)
    _step_case(orc, pad, 3, 0, 1, seed=28)       # the last rank holds only padding
    _step_case(orc, pad, 1, 0, 1, seed=29)
    pad.free()


def test_empty_range_touches_nothing():
    plan = zs.zs_flatten_plan([5000], world=4)
    S = plan.S
    st = [guarded(np.full(S, 0.5, np.float32)) for _ in range(3)]
    full = guarded(np.full(plan.P_pad, 0x1234, np.uint16))
    g = [to_dev(synth.fill(S, seed=30, rank=j, step=1, bf16=True)) for j in range(4)]
    for lo in (0, 17, S):
        zs.zs_shard_step(plan, 2, lo, lo, g, zs.ZS_BF16, *[x[1] for x in st], full[1],
                         zs.ZS_BF16, HP, 1)
    torch.cuda.synchronize()
    for whole, inner in st:
        assert bool((inner.view(torch.float32) == 0.5).all()) and intact(whole)
    assert bool((full[1].view(torch.int16) == 0x1234).all()) and intact(full[0])
    plan.free()


@pytest.mark.parametrize("lo,hi", [(0, 8 * 2048), (0, 8 * 2048 - 1), (1, 8 * 2048 + 3),
                                   (2048, 10 * 2048), (5, 9 * 2048 + 7)])
def test_staged_boundary_ranges(orc, lo, hi):
    """N = 16 bf16 slices (2048-element tiles) with the step path forced to
    staged: exactly 8 whole tiles runs the staged kernel, one element or one
    tile fewer falls back to the register-streaming kernel; both equal the
    oracle."""
    N = 16
    plan = zs.zs_flatten_plan([N * 10 * 2048], world=N, align_elems=128)
    assert plan.S == 10 * 2048
    _step_case(orc, plan, 9, lo, hi, seed=31, path=zs.STEP_PATH_STAGED)
    plan.free()


def test_buffers_same_as_list():
    """Slices passed as a zs.Buffers (marshalled once) give the same bits as
    the same slices passed as a list, for the step and the gather."""
    N = 64
    plan = zs.zs_flatten_plan([N * 5000], world=N, align_elems=16)
    S = plan.S
    g = [to_dev(synth.fill(S, seed=33, rank=j, step=1, bf16=True)) for j in range(N)]
    outs = []
    for slices in (g, zs.Buffers(g)):
        st = [to_dev(synth.fill(S, seed=33, stream=synth.STREAM_MASTER, sigma=0.02)),
              torch.zeros(S, device=DEV), torch.zeros(S, device=DEV)]
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        for t in (1, 2):
            zs.zs_shard_step(plan, 3, 0, S, slices, zs.ZS_BF16, *st, full, zs.ZS_BF16, HP, t)
        gathered = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        zs.zs_gather_assemble(plan, 0, slices, gathered, zs.ZS_BF16)
        torch.cuda.synchronize()
        outs.append([x.cpu().numpy().tobytes() for x in st + [full, gathered]])
    assert outs[0] == outs[1]
    plan.free()
