"""Both step kernels against the oracle: the register-streaming kernel and the
staged kernel (bulk asynchronous copies of 2048- or 1024-element tiles into
shared memory), each forced with zs_set_step_path, on ranges long enough for
the staged kernel (whole tiles plus ragged ends), every dtype pair, N up to 64,
with clipping, a skipped step and gradient accumulation; guard bands around
every buffer. The two kernels must give the oracle's bits."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import (DEV, ZS_OF, assert_params_close, assert_state_close, oracle_hp,
                      to_dev, to_host)
from synth.workloads import GPT2_SMALL
from test_gpu_parity import guarded, guards_intact

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture
def path(request):
    old = zs.zs_set_step_path(request.param)
    yield request.param
    zs.zs_set_step_path(old)


@pytest.mark.parametrize("path", [1, 2], indirect=True, ids=["direct", "staged"])
@pytest.mark.parametrize("seed", range(10))
def test_long_ranges_match_oracle(orc, path, seed):
    rng = np.random.default_rng(7100 + seed)
    N = int(rng.choice([1, 2, 3, 4, 8, 12, 16]))
    S0 = int(rng.integers(20_000, 300_000))
    plan = zs.zs_flatten_plan([N * S0 - int(rng.integers(0, 100))], world=N, align_elems=128)
    S, P = plan.S, plan.P
    rank = int(rng.integers(0, N))
    lo = int(rng.integers(0, 3000))
    hi = S - int(rng.integers(0, 3000))
    gdt = oracle.BF16 if seed % 3 else oracle.FP32
    pdt = [oracle.BF16, oracle.FP24, oracle.FP32][seed % 3]
    eb = oracle.ELEM_BYTES[pdt]
    bf16 = gdt == oracle.BF16
    master0 = synth.fill(S, index0=rank * S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02,
                         p_limit=P)
    o_st = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(plan.P_pad * eb, np.uint8)
    bufs = [guarded(S * 4, x) for x in o_st]
    full_whole, full = guarded(plan.P_pad * eb, o_full)
    for t in (1, 2):
        g_host = [synth.fill(S, index0=rank * S, seed=seed, rank=j, step=t, p_limit=P, bf16=bf16)
                  for j in range(N)]
        g_dev = [guarded(g.nbytes, g) for g in g_host]
        zs.zs_shard_step(plan, rank, lo, hi, [g[1] for g in g_dev],
                         zs.ZS_BF16 if bf16 else zs.ZS_FP32, bufs[0][1], bufs[1][1], bufs[2][1],
                         full, ZS_OF[pdt], HP, t)
        orc.shard_step(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=g_host, master=o_st[0],
                       m=o_st[1], v=o_st[2], full_flat=o_full, param_dtype=pdt, t=t,
                       **oracle_hp(HP))
        zs.zs_check_device_error()
        for name, (whole, inner), ref in zip(("master", "m", "v"), bufs, o_st):
            assert assert_state_close(to_host(inner, np.float32), ref, name) == 0, name
            assert guards_intact(whole), name
        got = to_host(full, np.uint8)
        assert assert_params_close(got, o_full, pdt) == 0
        assert np.array_equal(got, o_full)
        assert guards_intact(full_whole)
        for whole, _ in g_dev:
            assert guards_intact(whole)
    plan.free()


@pytest.mark.parametrize("path", [1, 2], indirect=True, ids=["direct", "staged"])
def test_clip_skip_and_accumulation(orc, path):
    """Clipped step (coefficient from device memory), a skipped step, and an
    accumulated step over G = 3 micro-steps, N = 8, S = 200,064."""
    N = 8
    plan = zs.zs_flatten_plan([N * 200_000], world=N, align_elems=128)
    S, P = plan.S, plan.P
    rank = 3
    st0 = synth.fill(S, index0=rank * S, seed=4, stream=synth.STREAM_MASTER, sigma=0.02,
                     p_limit=P)
    o = [st0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    d = [to_dev(x.copy()) for x in o]
    o_full = np.zeros(plan.P_pad, np.uint16)
    d_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    coef = torch.tensor([0.37], dtype=torch.float32, device=DEV)
    skip0 = torch.zeros(1, dtype=torch.int32, device=DEV)
    skip1 = torch.ones(1, dtype=torch.int32, device=DEV)

    def grads(t, k=0):
        return [synth.fill(S, index0=rank * S, seed=4, rank=j, step=10 * t + k, p_limit=P,
                           bf16=True) for j in range(N)]

    # t = 1: clipped
    g = grads(1)
    zs.zs_shard_step_clipped(plan, rank, 0, S, [to_dev(x) for x in g], zs.ZS_BF16, *d, d_full,
                             zs.ZS_BF16, HP, 1, coef=coef, skip=skip0)
    orc.shard_step_clipped(world=N, rank=rank, S=S, lo=0, hi=S, grads=g, master=o[0], m=o[1],
                           v=o[2], full_flat=o_full, coef=np.float32(0.37), skip=0, t=1,
                           **oracle_hp(HP))
    # t = 2: skipped (nothing changes)
    g = grads(2)
    zs.zs_shard_step_clipped(plan, rank, 0, S, [to_dev(x) for x in g], zs.ZS_BF16, *d, d_full,
                             zs.ZS_BF16, HP, 2, coef=coef, skip=skip1)
    # t = 2 again: G = 3 micro-steps
    acc = torch.empty(S, dtype=torch.float32, device=DEV)
    o_acc = np.zeros(S, np.float32)
    for k in range(3):
        g = grads(3, k)
        dg = [to_dev(x) for x in g]
        if k < 2:
            zs.zs_grad_accumulate(plan, rank, 0, S, dg, zs.ZS_BF16, acc, k == 0)
            orc.grad_accumulate(world=N, S=S, lo=0, hi=S, grads=g, accum=o_acc, first=k == 0)
        else:
            zs.zs_shard_step_accumulated(plan, rank, 0, S, dg, zs.ZS_BF16, acc, 3, *d, d_full,
                                         zs.ZS_BF16, HP, 2)
            orc.shard_step_accumulated(world=N, rank=rank, S=S, lo=0, hi=S, grads=g, accum=o_acc,
                                       micro_steps=3, master=o[0], m=o[1], v=o[2],
                                       full_flat=o_full, t=2, **oracle_hp(HP))
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    for name, x, ref in zip(("master", "m", "v"), d, o):
        assert assert_state_close(to_host(x, np.float32), ref, name) == 0
    assert np.array_equal(to_host(d_full, np.uint16), o_full)
    plan.free()


def test_both_kernels_identical_on_gpt2_small():
    """The GPT-2-small shard (S = 15,555,072, N = 8, rank 6), three steps
    through each kernel from the same inputs: identical bits everywhere."""
    w = GPT2_SMALL
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    rank = 6
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    outs = []
    for path in (1, 2):
        old = zs.zs_set_step_path(path)
        try:
            st = [torch.empty(S, dtype=torch.float32, device=DEV) for _ in range(3)]
            synth.fill_device(st[0].data_ptr(), S, index0=rank * S, seed=w.seed,
                              stream=synth.STREAM_MASTER, sigma=w.master_sigma, p_limit=P,
                              cuda_stream=stream)
            st[1].zero_()
            st[2].zero_()
            full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
            for t in (1, 2, 3):
                for j, g in enumerate(grads):
                    synth.fill_device(g.data_ptr(), S, index0=rank * S, seed=w.seed, rank=j,
                                      step=t, sigma=w.grad_sigma, p_limit=P, bf16=True,
                                      cuda_stream=stream)
                zs.zs_shard_step(plan, rank, 0, S, grads, zs.ZS_BF16, *st, full, zs.ZS_BF16, HP,
                                 t)
            torch.cuda.synchronize()
            outs.append([x.view(torch.int32) for x in st] + [full])
        finally:
            zs.zs_set_step_path(old)
    zs.zs_check_device_error()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    plan.free()


def test_step_path_switch():
    old = zs.zs_set_step_path(2)
    assert zs.zs_set_step_path(1) == 2
    assert zs.zs_set_step_path(old) == 1
    with pytest.raises(ValueError):
        zs.zs_set_step_path(3)
    assert zs.zs_set_step_path(old) == old


def test_bounded_wait_runs_out_and_the_context_survives(orc):
    """A wait that nothing satisfies gives up after its poll limit, sets the
    timeout bit of the device error word (ZS_ERR_TIMEOUT on the host), and the
    context stays usable: a staged step afterwards matches the oracle."""
    zs.zs_check_device_error()   # start from a clear error word
    zs.zs_selftest_wait_timeout(1000)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_check_device_error()
    assert e.value.status == zs.ZS_ERR_TIMEOUT
    zs.zs_check_device_error()   # read and cleared
    old = zs.zs_set_step_path(2)
    try:
        N, S0 = 4, 40_000
        plan = zs.zs_flatten_plan([N * S0], world=N, align_elems=128)
        S = plan.S
        g = [synth.fill(S, seed=3, rank=j, step=1, bf16=True, p_limit=N * S) for j in range(N)]
        master = synth.fill(S, seed=3, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=N * S)
        o = [master.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
        d = [to_dev(x.copy()) for x in o]
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        o_full = np.zeros(plan.P_pad, np.uint16)
        zs.zs_shard_step(plan, 0, 0, S, [to_dev(x) for x in g], zs.ZS_BF16, *d, full, zs.ZS_BF16,
                         HP, 1)
        orc.shard_step(world=N, rank=0, S=S, lo=0, hi=S, grads=g, master=o[0], m=o[1], v=o[2],
                       full_flat=o_full, t=1, **oracle_hp(HP))
        zs.zs_check_device_error()
        for x, ref, name in zip(d, o, ("master", "m", "v")):
            assert assert_state_close(to_host(x, np.float32), ref, name) == 0
        assert np.array_equal(to_host(full, np.uint16), o_full)
        plan.free()
    finally:
        zs.zs_set_step_path(old)


@pytest.mark.parametrize("N,bf16", [(2, True), (3, True), (4, True), (8, True), (16, True),
                                    (2, False), (8, False)])
def test_large_ranges_identical_bits(N, bf16):
    """S = 2^25 (16,384 tiles; every stage of every block reused hundreds of
    times), two steps through each kernel from the same inputs: master, m, v
    and the parameter slot identical bit for bit. A stage released too early
    or a copy landing late would show here."""
    S = 1 << 25
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
    assert plan.S == S
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(S * (2 if bf16 else 4), dtype=torch.uint8, device=DEV) for _ in range(N)]
    outs = []
    for path in (1, 2):
        old = zs.zs_set_step_path(path)
        try:
            st = [torch.empty(S, dtype=torch.float32, device=DEV) for _ in range(3)]
            synth.fill_device(st[0].data_ptr(), S, seed=11, stream=synth.STREAM_MASTER, sigma=0.02,
                              cuda_stream=stream)
            st[1].zero_()
            st[2].zero_()
            full = torch.zeros(N * S, dtype=torch.int16, device=DEV)
            for t in (1, 2):
                for j, g in enumerate(grads):
                    synth.fill_device(g.data_ptr(), S, seed=11, rank=j, step=t, bf16=bf16,
                                      cuda_stream=stream)
                zs.zs_shard_step(plan, 0, 0, S, grads, zs.ZS_BF16 if bf16 else zs.ZS_FP32, *st,
                                 full, zs.ZS_BF16, HP, t)
            torch.cuda.synchronize()
            outs.append([x.view(torch.int32) for x in st] + [full.narrow(0, 0, S)])
        finally:
            zs.zs_set_step_path(old)
    zs.zs_check_device_error()
    for name, a, b in zip(("master", "m", "v", "params"), *outs):
        assert torch.equal(a, b), name
    plan.free()


@pytest.mark.parametrize("path", [1, 2], indirect=True, ids=["direct", "staged"])
@pytest.mark.parametrize("pdt", [oracle.BF16, oracle.FP24, oracle.FP32], ids=["bf16", "fp24", "fp32"])
def test_step_to_shard_matches_oracle(orc, path, pdt):
    """zs_shard_step_to_shard writes the parameters into a shard buffer of its
    own (S elements, guard bands around it): its bytes equal the oracle's slot,
    the state matches, and nothing outside [lo, hi) of the shard is written."""
    N, rank = 4, 2
    plan = zs.zs_flatten_plan([N * 60_000 - 37], world=N, align_elems=128)
    S, P = plan.S, plan.P
    lo, hi = 1111, S - 777
    eb = oracle.ELEM_BYTES[pdt]
    master0 = synth.fill(S, index0=rank * S, seed=8, stream=synth.STREAM_MASTER, sigma=0.02,
                         p_limit=P)
    o = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    d = [guarded(S * 4, x) for x in o]
    o_full = np.zeros(plan.P_pad * eb, np.uint8)
    shard_whole, shard = guarded(S * eb, np.zeros(S * eb, np.uint8))
    for t in (1, 2):
        g = [synth.fill(S, index0=rank * S, seed=8, rank=j, step=t, p_limit=P, bf16=True)
             for j in range(N)]
        zs.zs_shard_step_to_shard(plan, rank, lo, hi, [to_dev(x) for x in g], zs.ZS_BF16,
                                  d[0][1], d[1][1], d[2][1], shard, ZS_OF[pdt], HP, t)
        orc.shard_step(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=g, master=o[0], m=o[1],
                       v=o[2], full_flat=o_full, param_dtype=pdt, t=t, **oracle_hp(HP))
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    for name, (whole, inner), ref in zip(("master", "m", "v"), d, o):
        assert assert_state_close(to_host(inner, np.float32), ref, name) == 0
        assert guards_intact(whole)
    got = to_host(shard, np.uint8)
    assert np.array_equal(got, o_full[rank * S * eb:(rank + 1) * S * eb])
    assert guards_intact(shard_whole)
    plan.free()


@pytest.mark.parametrize("path", [2], indirect=True, ids=["staged"])
@pytest.mark.parametrize("N,bf16", [(20, True), (32, True), (48, True), (16, False), (24, False),
                                    (64, True), (32, False)],
                         ids=["bf16x20-tile2048", "bf16x32-tile1024", "bf16x48-tile1024",
                              "fp32x16-tile1024", "fp32x24-tile1024", "bf16x64-unstaged",
                              "fp32x32-unstaged"])
@pytest.mark.parametrize("pdt", [oracle.BF16, oracle.FP24, oracle.FP32], ids=["bf16", "fp24", "fp32"])
def test_narrow_tiles_match_oracle(orc, path, N, bf16, pdt):
    """Many slices, the staged kernel forced: 2048-element tiles while two
    stages of them fit in shared memory, else 1024-element tiles, else (no
    tile fits) the register-streaming kernel; over a ragged range, the plain
    step then a clipped accumulated step, against the oracle bit for bit with
    guard bands."""
    S0 = 23_000
    plan = zs.zs_flatten_plan([N * S0], world=N, align_elems=128)
    S, P = plan.S, plan.P
    rank, lo, hi = N // 2, 301, S - 77
    eb = oracle.ELEM_BYTES[pdt]
    master0 = synth.fill(S, index0=rank * S, seed=N, stream=synth.STREAM_MASTER, sigma=0.02,
                         p_limit=P)
    o_st = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(plan.P_pad * eb, np.uint8)
    bufs = [guarded(S * 4, x) for x in o_st]
    full_whole, full = guarded(plan.P_pad * eb, o_full)
    gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
    acc = (np.random.default_rng(N).standard_normal(S) * 1e-3).astype(np.float32)
    acc_whole, d_acc = guarded(S * 4, acc)
    coef = torch.tensor([0.625], dtype=torch.float32, device=DEV)
    skip = torch.zeros(1, dtype=torch.int32, device=DEV)
    for t in (1, 2):
        g_host = [synth.fill(S, index0=rank * S, seed=N, rank=j, step=t, p_limit=P, bf16=bf16)
                  for j in range(N)]
        g_dev = [guarded(g.nbytes, g) for g in g_host]
        dev_slices = [g[1] for g in g_dev]
        if t == 1:
            zs.zs_shard_step(plan, rank, lo, hi, dev_slices, gdt, *[b[1] for b in bufs], full,
                             ZS_OF[pdt], HP, t)
            orc.shard_step(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=g_host, master=o_st[0],
                           m=o_st[1], v=o_st[2], full_flat=o_full, param_dtype=pdt, t=t,
                           **oracle_hp(HP))
        else:
            zs.zs_shard_step_accumulated_clipped(plan, rank, lo, hi, dev_slices, gdt, d_acc, 3,
                                                 *[b[1] for b in bufs], full, ZS_OF[pdt], HP, t,
                                                 coef=coef, skip=skip)
            orc.shard_step_accumulated_clipped(world=N, rank=rank, S=S, lo=lo, hi=hi,
                                               grads=g_host, accum=acc, micro_steps=3,
                                               master=o_st[0], m=o_st[1], v=o_st[2],
                                               full_flat=o_full, coef=np.float32(0.625), skip=0,
                                               param_dtype=pdt, t=t, **oracle_hp(HP))
        zs.zs_check_device_error()
        for name, (whole, inner), ref in zip(("master", "m", "v"), bufs, o_st):
            got = to_host(inner, np.float32)
            assert assert_state_close(got, ref, name) == 0, name
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), name
            assert guards_intact(whole), name
        got = to_host(full, np.uint8)
        assert assert_params_close(got, o_full, pdt) == 0
        assert np.array_equal(got, o_full)
        assert guards_intact(full_whole) and guards_intact(acc_whole)
        for whole, _ in g_dev:
            assert guards_intact(whole)
    plan.free()
