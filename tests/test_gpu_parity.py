"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs. fp32 master/m/v within 1e-6 max relative error, low-
precision parameters within 1 ulp, layout and gather bit-exact (bit-exact is
also asserted for the fp32 states: the op sequence is the same IEEE one)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import (DEV, ZS_OF, assert_params_close, assert_state_close, dev_fill,
                      oracle_hp, to_dev, to_host)
from synth.workloads import GPT2_SMALL, LLAMA_7B, QWEN25_3B, TINY

pytestmark = pytest.mark.gpu

CANARY = 0x5A


def guarded(nbytes, fill=None, front=256):
    """A device byte buffer with guard bands of CANARY on both sides (``front``
    bytes before, 256 after); returns (whole, interior). front = 256 gives a
    32-byte aligned interior, 272 one that is only 16-byte aligned."""
    whole = torch.full((front + nbytes + 256,), CANARY, dtype=torch.uint8, device=DEV)
    inner = whole.narrow(0, front, nbytes)
    if fill is not None:
        inner.copy_(torch.from_numpy(np.ascontiguousarray(fill).view(np.uint8)).to(DEV))
    whole.zs_front = front
    return whole, inner


def guards_intact(whole):
    front = whole.zs_front
    g = torch.cat([whole[:front], whole[whole.numel() - 256:]])
    return bool((g == CANARY).all())


def random_case(seed):
    rng = np.random.default_rng(seed)
    world = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 64]))
    k = int(rng.integers(1, 7))
    numels = [int(x) for x in rng.integers(1, 4000 if world < 16 else 1500, size=k)]
    ties = [-1] * k
    if k >= 3:
        numels[-1] = numels[0]
        ties[-1] = 0
    align = int(rng.choice([128, 128, 8, 1]))
    gdt = oracle.BF16 if rng.random() < 0.7 else oracle.FP32
    pdt = int(rng.choice([oracle.BF16, oracle.BF16, oracle.FP24, oracle.FP32]))
    return rng, world, numels, ties, align, gdt, pdt


@pytest.mark.parametrize("seed", range(24))
def test_random_small_cases(orc, seed):
    """Random parameter lists (ties, odd sizes), N in 1..64, bf16/fp32 incoming
    slices, bf16/3-byte/fp32 parameters, a random rank and a ragged [lo, hi),
    three steps; outputs and 256-byte guard bands around every buffer."""
    rng, N, numels, ties, align, gdt, pdt = random_case(seed)
    plan = zs.zs_flatten_plan(numels, ties, world=N, align_elems=align)
    o_plan = orc.plan(numels, ties, world=N, align=align)
    S, P, P_pad = plan.S, plan.P, plan.P_pad
    assert (S, P, P_pad) == (o_plan["S"], o_plan["P"], o_plan["P_pad"])
    rank = int(rng.integers(0, N))
    lo = int(rng.integers(0, max(1, S // 3)))
    hi = int(rng.integers(max(lo, 2 * S // 3), S + 1))
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    eb = oracle.ELEM_BYTES[pdt]
    master0 = synth.fill(S, index0=rank * S, seed=seed, stream=synth.STREAM_MASTER,
                         sigma=0.02, p_limit=P)
    o_state = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(P_pad * eb, np.uint8)
    # Some seeds place one buffer only 16-byte aligned: the 16-byte vector path.
    fronts = [256] * (N + 4)
    if seed % 3 == 1:
        fronts[int(rng.integers(0, N + 4))] = 272
    bufs = [guarded(S * 4, o_state[k], fronts[N + k]) for k in range(3)]
    full_whole, full = guarded(P_pad * eb, o_full, fronts[N + 3])
    bf16 = gdt == oracle.BF16
    for t in (1, 2, 3):
        g_host = [synth.fill(S, index0=rank * S, seed=seed, rank=j, step=t, p_limit=P,
                             bf16=bf16) for j in range(N)]
        g_dev = [guarded(g.nbytes, g, fronts[j]) for j, g in enumerate(g_host)]
        zs.zs_shard_step(plan, rank, lo, hi, [g[1] for g in g_dev],
                         zs.ZS_BF16 if bf16 else zs.ZS_FP32, bufs[0][1], bufs[1][1],
                         bufs[2][1], full, ZS_OF[pdt], hp, t)
        orc.shard_step(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=g_host, master=o_state[0],
                       m=o_state[1], v=o_state[2], full_flat=o_full, param_dtype=pdt, t=t,
                       **oracle_hp(hp))
        zs.zs_check_device_error()
        for name, (whole, inner), ref in zip(("master", "exp_avg", "exp_avg_sq"), bufs, o_state):
            got = to_host(inner, np.float32)
            assert assert_state_close(got, ref, name) == 0, f"{name} not bit-exact"
            assert guards_intact(whole), f"{name} guard band overwritten"
        got_full = to_host(full, np.uint8)
        assert assert_params_close(got_full, o_full, pdt) == 0
        assert np.array_equal(got_full, o_full), "flat buffer differs outside the own slot"
        assert guards_intact(full_whole)
        for whole, _ in g_dev:
            assert guards_intact(whole)
    plan.free()


def test_tiny_all_ranks_then_gather_equals_ddp(orc):
    """The tiny 2-layer transformer list (N = 4, ZeRO-1 layout), 3 steps: each
    rank's GPU step, then the GPU gather, equals the oracle's unsharded DDP
    AllReduce + AdamW step bit for bit."""
    w = TINY
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P, P_pad = plan.world, plan.S, plan.P, plan.P_pad
    hp = w.hparams
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    ddp = dict(master=master0.copy(), m=np.zeros(P_pad, np.float32),
               v=np.zeros(P_pad, np.float32), params=np.zeros(P_pad, np.uint16))
    d_master = [to_dev(master0[r * S:(r + 1) * S].copy()) for r in range(N)]
    d_m = [torch.zeros(S, dtype=torch.float32, device=DEV) for _ in range(N)]
    d_v = [torch.zeros(S, dtype=torch.float32, device=DEV) for _ in range(N)]
    d_full = [torch.zeros(P_pad, dtype=torch.int16, device=DEV) for _ in range(N)]
    for t in range(1, w.steps + 1):
        local = [synth.fill(P_pad, seed=w.seed, rank=j, step=t, sigma=w.grad_sigma, p_limit=P,
                            bf16=True) for j in range(N)]
        orc.ddp_step(world=N, P_pad=P_pad, local_grads=local, **ddp, t=t, **oracle_hp(hp))
        d_local = [to_dev(x) for x in local]
        for r in range(N):
            slices = [d_local[j].narrow(0, r * S, S) for j in range(N)]
            zs.zs_shard_step(plan, r, 0, S, slices, zs.ZS_BF16, d_master[r], d_m[r], d_v[r],
                             d_full[r], zs.ZS_BF16, hp, t)
        for r in range(N):
            own = [d_full[j].narrow(0, j * S, S) for j in range(N)]
            zs.zs_gather_assemble(plan, r, own, d_full[r], zs.ZS_BF16)
        torch.cuda.synchronize()
        for r in range(N):
            assert np.array_equal(to_host(d_full[r], np.uint16), ddp["params"]), f"t={t} r={r}"
        for name, dl in (("master", d_master), ("m", d_m), ("v", d_v)):
            got = np.concatenate([to_host(x, np.float32) for x in dl])
            assert assert_state_close(got, ddp[name], name) == 0
    plan.free()


def test_gpt2_small_buckets_ten_steps(orc):
    """GPT-2-small list, N = 8, ZeRO-2 with 25M-element buckets: rank 3's step
    as per-bucket sub-range calls, 10 steps, against the oracle's whole-shard
    step (bucketed == whole is pinned on the oracle side)."""
    w = GPT2_SMALL
    rank = 3
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align,
                              bucket_elems=w.bucket_elems)
    N, S, P = plan.world, plan.S, plan.P
    assert plan.n_buckets == 5
    ranges = [zs.zs_plan_bucket(plan, b, rank) for b in range(plan.n_buckets)]
    ranges = [(lo, hi) for lo, hi in ranges if hi > lo]
    assert sum(hi - lo for lo, hi in ranges) == S and len(ranges) >= 2
    hp = w.hparams
    d_master = dev_fill(S, bf16=False, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                        sigma=w.master_sigma, p_limit=P)
    d_m = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_v = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    o_master = synth.fill(S, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                          sigma=w.master_sigma, p_limit=P)
    assert np.array_equal(to_host(d_master, np.float32), o_master), "device/host generators"
    o_m, o_v = np.zeros(S, np.float32), np.zeros(S, np.float32)
    o_full = np.zeros(plan.P_pad, np.uint16)
    d_grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    for t in range(1, w.steps + 1):
        for j in range(N):
            synth.fill_device(d_grads[j].data_ptr(), S, index0=rank * S, seed=w.seed, rank=j,
                              step=t, sigma=w.grad_sigma, p_limit=P, bf16=True,
                              cuda_stream=torch.cuda.current_stream().cuda_stream)
        for lo, hi in ranges:
            zs.zs_shard_step(plan, rank, lo, hi, d_grads, zs.ZS_BF16, d_master, d_m, d_v,
                             d_full, zs.ZS_BF16, hp, t)
        g_host = [synth.fill(S, index0=rank * S, seed=w.seed, rank=j, step=t,
                             sigma=w.grad_sigma, p_limit=P, bf16=True) for j in range(N)]
        orc.shard_step(world=N, rank=rank, S=S, lo=0, hi=S, grads=g_host, master=o_master,
                       m=o_m, v=o_v, full_flat=o_full, t=t, **oracle_hp(hp))
    torch.cuda.synchronize()
    for name, d, ref in (("master", d_master, o_master), ("m", d_m, o_m), ("v", d_v, o_v)):
        assert assert_state_close(to_host(d, np.float32), ref, name) == 0
    got = to_host(d_full, np.uint16)
    assert assert_params_close(got, o_full, oracle.BF16) == 0
    assert np.array_equal(got, o_full)
    plan.free()


def _full_size_sampled(orc, w, steps, rank, n_samples=60_000):
    """Full-size step in the benchmark's launch configuration; sampled elements
    recomputed by the oracle from regenerated inputs; the cast checked on every
    element via a library conversion."""
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    hp = w.hparams
    kw = dict(seed=w.seed, sigma=w.grad_sigma, p_limit=P, outlier_frac=w.outlier_frac,
              outlier_scale=w.outlier_scale, bf16=True)
    d_master = dev_fill(S, bf16=False, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                        sigma=w.master_sigma, p_limit=P)
    d_m = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_v = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    d_grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    rng = np.random.default_rng(17)
    idx = np.unique(np.concatenate([
        rng.integers(0, S, size=n_samples), np.arange(0, 64), np.arange(S - 64, S),
        np.arange(S // 2 - 8, S // 2 + 8)])).astype(np.int64)
    gidx = idx + rank * S
    o_master = synth.at(gidx, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                        p_limit=P)
    K = idx.size
    o_m, o_v = np.zeros(K, np.float32), np.zeros(K, np.float32)
    o_full = np.zeros(K * N, np.uint16)
    for t in range(1, steps + 1):
        for j in range(N):
            synth.fill_device(d_grads[j].data_ptr(), S, index0=rank * S, rank=j, step=t,
                              cuda_stream=torch.cuda.current_stream().cuda_stream, **kw)
        zs.zs_shard_step(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_master, d_m, d_v, d_full,
                         zs.ZS_BF16, hp, t)
        g_host = [synth.at(gidx, rank=j, step=t, **kw) for j in range(N)]
        orc.shard_step(world=N, rank=0, S=K, lo=0, hi=K, grads=g_host, master=o_master, m=o_m,
                       v=o_v, full_flat=o_full, t=t, **oracle_hp(hp))
    torch.cuda.synchronize()
    ti = torch.from_numpy(idx).to(DEV)
    for name, d, ref in (("master", d_master, o_master), ("m", d_m, o_m), ("v", d_v, o_v)):
        assert assert_state_close(d[ti].cpu().numpy(), ref, name) == 0
    slot = d_full.narrow(0, rank * S, S)
    got = slot[ti].cpu().numpy().view(np.uint16)
    assert assert_params_close(got, o_full[:K], oracle.BF16) == 0
    # Every element: the slot holds the nearest-even bf16 of the master.
    ref_all = d_master.to(torch.bfloat16).view(torch.int16)
    assert bool((slot == ref_all).all())
    # Other slots untouched; the tail pad (if in this shard) stays zero.
    assert int(d_full.narrow(0, 0, rank * S).count_nonzero()) == 0
    if (rank + 1) * S > P:
        pad0 = max(P - rank * S, 0)
        assert int(d_master[pad0:].count_nonzero()) == 0 and int(slot[pad0:].count_nonzero()) == 0
    plan.free()


def test_qwen25_3b_full_size_sampled(orc):
    _full_size_sampled(orc, QWEN25_3B, steps=3, rank=2)


def test_llama_7b_full_size_sampled(orc):
    _full_size_sampled(orc, LLAMA_7B, steps=2, rank=5)


def test_device_generator_matches_host():
    for bf16 in (True, False):
        for kw in (dict(seed=0, rank=3, step=7, sigma=1e-3), dict(seed=5, stream=1, sigma=0.02),
                   dict(seed=1, rank=1, step=2, sigma=1e-3, outlier_frac=0.01,
                        outlier_scale=100.0)):
            n = 300_001
            d = dev_fill(n, bf16=bf16, index0=12345, p_limit=12345 + n - 17, **kw)
            h = synth.fill(n, index0=12345, p_limit=12345 + n - 17, bf16=bf16, **kw)
            assert np.array_equal(to_host(d, h.dtype), h)


@pytest.mark.parametrize("pdt", [oracle.BF16, oracle.FP24, oracle.FP32])
def test_gather_assemble(orc, pdt):
    """Every other rank's shard lands in its slot bit for bit; the own slot, NULL
    entries and sources already in place are skipped; views follow offsets."""
    numels = [777, 1000, 333, 777, 4096]
    ties = [-1, -1, -1, 0, -1]
    N = 5
    plan = zs.zs_flatten_plan(numels, ties, world=N)
    S, P_pad = plan.S, plan.P_pad
    eb = oracle.ELEM_BYTES[pdt]
    rng = np.random.default_rng(pdt)
    shards = [rng.integers(0, 256, size=S * eb, dtype=np.uint8) for _ in range(N)]
    rank = 2
    init = rng.integers(0, 256, size=P_pad * eb, dtype=np.uint8)
    full_whole, full = guarded(P_pad * eb, init)
    srcs = [to_dev(s) for s in shards]
    srcs[4] = None                                     # NULL: slot 4 untouched
    srcs[1] = full.narrow(0, 1 * S * eb, S * eb)       # already in place: skipped
    views = zs.zs_gather_assemble(plan, rank, srcs, full, ZS_OF[pdt])
    torch.cuda.synchronize()
    expect = init.copy()
    orc.gather(world=N, S=S, elem_size=eb,
               shards=[shards[0], None, None, shards[3], None], full_flat=expect)
    assert np.array_equal(to_host(full, np.uint8), expect)
    assert guards_intact(full_whole)
    offs = zs.zs_plan_offsets(plan)
    assert [v - full.data_ptr() for v in views] == [o * eb for o in offs]
    assert views[3] == views[0]
    plan.free()


def test_nan_inf_propagate(orc):
    """NaN and infinite gradients propagate per IEEE into m, v and the master
    (no trap), exactly as on the CPU."""
    N, S = 4, 1024
    plan = zs.zs_flatten_plan([S * N], world=N)
    g = [synth.fill(S, seed=1, rank=j, step=1, bf16=True) for j in range(N)]
    g[1][5] = 0x7FC0      # NaN
    g[2][9] = 0x7F80      # +inf
    g[3][9] = 0xFF80      # -inf -> inf + -inf = NaN
    g[0][100] = 0x7F80    # +inf alone
    g[0][200] = 0x7F7F    # largest finite bf16: its square overflows v
    master = synth.fill(S, seed=1, stream=synth.STREAM_MASTER, sigma=0.02)
    o = [master.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_full = np.zeros(S * N, np.uint16)
    d = [to_dev(x.copy()) for x in o]
    d_full = torch.zeros(S * N, dtype=torch.int16, device=DEV)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    zs.zs_shard_step(plan, 0, 0, S, [to_dev(x) for x in g], zs.ZS_BF16, *d, d_full,
                     zs.ZS_BF16, hp, 1)
    orc.shard_step(world=N, rank=0, S=S, lo=0, hi=S, grads=g, master=o[0], m=o[1], v=o[2],
                   full_flat=o_full, t=1, **oracle_hp(hp))
    for name, dt, ref in zip(("master", "m", "v"), d, o):
        assert_state_close(to_host(dt, np.float32), ref, name)
    assert np.isnan(o[0][5]) and np.isnan(o[0][9])
    assert_params_close(to_host(d_full, np.uint16), o_full, oracle.BF16)
    plan.free()


def test_side_stream_and_validation_off(orc):
    """Work enqueued on a non-default stream, and with pointer validation off,
    gives the same bits."""
    N, S = 8, 4096 + 128
    plan = zs.zs_flatten_plan([S * N - 5], world=N)
    S = plan.S
    g = [synth.fill(S, seed=4, rank=j, step=1, bf16=True) for j in range(N)]
    master = synth.fill(S, seed=4, stream=synth.STREAM_MASTER, sigma=0.02)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    outs = []
    for level in (1, 0):
        old = zs.zs_set_validation(level)
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                d = [to_dev(master.copy()), torch.zeros(S, device=DEV), torch.zeros(S, device=DEV)]
                full = torch.zeros(S * N, dtype=torch.int16, device=DEV)
                zs.zs_shard_step(plan, 1, 0, S, [to_dev(x) for x in g], zs.ZS_BF16, *d, full,
                                 zs.ZS_BF16, hp, 1, stream=s)
            s.synchronize()
            outs.append([to_host(x, np.uint32) for x in d] + [to_host(full, np.uint16)])
        finally:
            zs.zs_set_validation(old)
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    plan.free()


def test_device_pointer_errors():
    """Rejected before any kernel runs: a buffer shorter than its extent, a host
    pointer, a misaligned pointer, overlapping outputs."""
    N, S = 4, 1024
    plan = zs.zs_flatten_plan([S * N], world=N)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    grads = [torch.zeros(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    st = [torch.zeros(S, device=DEV) for _ in range(3)]
    full = torch.zeros(S * N, dtype=torch.int16, device=DEV)

    def call(hi=S, **kw):
        a = dict(grad_slices=grads, master=st[0], exp_avg=st[1], exp_avg_sq=st[2], full_flat=full)
        a.update(kw)
        zs.zs_shard_step(plan, 0, 0, hi, a["grad_slices"], zs.ZS_BF16, a["master"],
                         a["exp_avg"], a["exp_avg_sq"], a["full_flat"], zs.ZS_BF16, hp, 1)

    call()  # the good call works
    # A master pointer 1 KiB before the end of its own 12 MiB allocation: the
    # shard needs 4 KiB, so the call is refused. Only elements [0, 8) are
    # asked for, so even a missed check could not write past the allocation.
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    big = torch.empty(3 * 1024 * 1024, dtype=torch.float32, device=DEV)
    near_end = big.data_ptr() + big.numel() * 4 - 1024
    with pytest.raises(zs.ZsError) as e:
        call(hi=8, master=near_end)
    assert e.value.status == zs.ZS_ERR_RANGE, str(e.value)
    del big
    host = torch.zeros(S)
    with pytest.raises(zs.ZsError) as e:
        call(hi=8, master=host.data_ptr())
    assert e.value.status == zs.ZS_ERR_INVAL
    with pytest.raises(zs.ZsError) as e:
        call(exp_avg=st[1].data_ptr() + 4)
    assert e.value.status == zs.ZS_ERR_ALIGN
    with pytest.raises(zs.ZsError) as e:
        call(exp_avg_sq=st[0])
    assert e.value.status == zs.ZS_ERR_INVAL
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    plan.free()
