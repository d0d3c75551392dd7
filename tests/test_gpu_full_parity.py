"""GPU parity over EVERY element of the named workloads at full size, for the
stated number of steps: the CUDA path through the C ABI, in the launch
configuration the benchmark times, against the CPU oracle run chunk by chunk
over the whole shard on every host core (tests/full_parity.py). master, m, v
and the parameter bytes are compared bit for bit (the gates, 1e-6 relative
for the fp32 state and 1 ulp for the parameters, are asserted as well).

Workloads (synth/workloads.py): GPT-2-small at N = 8 with ZeRO-2's 25M-element
buckets, every rank, 10 steps ("DeepSpeed ZeRO vs PyTorch FSDP2, measured"
uses the ZeRO-2 layout; the GPT-2-small list is the small configuration);
Qwen2.5-3B at N = 4, 15 steps ("DeepSpeed ZeRO vs PyTorch FSDP2, measured",
Chapter 2: Qwen2.5-3B on 4 GPUs, 15 steps); Llama-7B at N = 8 with 1 % of the
gradient entries scaled by 100, 10 steps ("ZeRO vs FSDP: A Rigorous
Dissection", §2.1-2.3: a 7B model at dp = 8); and the sweep's grid of N x
slice dtype x parameter dtype at 2^24 elements (every element) and 2^28
elements (sampled).

These tests run the oracle over billions of element-steps on the host (a few
minutes on 16 cores); the bounds-checked child process (test_gpu_bounds.py)
skips them and runs the sampled full-size tests of test_gpu_parity.py instead.
"""
import os

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from full_parity import CHUNK, bitwise_check, oracle_chunks, run_chunks
from gpu_util import (DEV, all_zero, assert_params_close, assert_state_close, dev_fill,
                      oracle_hp)
from synth.workloads import GPT2_SMALL, LLAMA_7B, QWEN25_3B, SWEEP_WORLDS

pytestmark = [
    pytest.mark.gpu,
    pytest.mark.skipif(os.environ.get("ZS_BOUNDS_CHECK") == "1",
                       reason="host oracle over every element runs in the ordinary suite"),
]

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _host(t, dtype):
    return t.cpu().numpy().view(dtype)


def _flat_workload(orc, w, rank, steps):
    """The whole-shard step of rank `rank`, `steps` steps, every element."""
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P, P_pad = plan.world, plan.S, plan.P, plan.P_pad
    o_plan = orc.plan(w.numels, w.tied_to, world=w.world, align=w.align)
    assert (S, P, P_pad) == (o_plan["S"], o_plan["P"], o_plan["P_pad"])
    grad_kw = dict(seed=w.seed, sigma=w.grad_sigma, outlier_frac=w.outlier_frac,
                   outlier_scale=w.outlier_scale, bf16=True)
    master_kw = dict(seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma)
    stream = torch.cuda.current_stream().cuda_stream
    d_master = dev_fill(S, bf16=False, index0=rank * S, p_limit=P, **master_kw)
    d_m = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_v = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_full = torch.zeros(P_pad, dtype=torch.int16, device=DEV)
    d_grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    for t in range(1, steps + 1):
        for j in range(N):
            synth.fill_device(d_grads[j].data_ptr(), S, index0=rank * S, rank=j, step=t,
                              p_limit=P, cuda_stream=stream, **grad_kw)
        zs.zs_shard_step(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_master, d_m, d_v, d_full,
                         zs.ZS_BF16, w.hparams, t)
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    del d_grads
    g_master, g_m, g_v = _host(d_master, np.float32), _host(d_m, np.float32), _host(d_v, np.float32)
    g_slot = _host(d_full.narrow(0, rank * S, S), np.uint8)
    # The other ranks' slots are untouched.
    assert all_zero(d_full.narrow(0, 0, rank * S))
    assert all_zero(d_full.narrow(0, (rank + 1) * S, P_pad - (rank + 1) * S))
    del d_master, d_m, d_v, d_full
    torch.cuda.empty_cache()
    check = bitwise_check(g_master, g_m, g_v, {oracle.BF16: g_slot})
    diff = oracle_chunks(orc, world=N, rank=rank, S=S, P=P, steps=steps, hp=w.hparams,
                         grad_kw=grad_kw, master_kw=master_kw, pdts=[oracle.BF16], check=check)
    assert diff == 0, f"{diff} elements differ in some bit (within the gates)"
    # The tail pad of the last shard stays zero (master, moments, parameters).
    if (rank + 1) * S > P:
        pad0 = max(P - rank * S, 0)
        assert not g_master[pad0:].any() and not g_m[pad0:].any() and not g_slot[2 * pad0:].any()
    plan.free()


def test_llama_7b_every_element_ten_steps(orc):
    """Llama-7B, N = 8, rank 5's shard (842,301,952 elements), 10 steps, with the
    1 % x 100 gradient outliers: every element bit for bit."""
    _flat_workload(orc, LLAMA_7B, rank=5, steps=LLAMA_7B.steps)


def test_qwen25_3b_every_element_fifteen_steps(orc):
    """Qwen2.5-3B, N = 4, the last rank's shard (771,484,672 elements), 15 steps:
    every element bit for bit."""
    _flat_workload(orc, QWEN25_3B, rank=3, steps=QWEN25_3B.steps)


def test_gpt2_small_every_rank_bucketed_ten_steps(orc):
    """GPT-2-small, N = 8, ZeRO-2 with 25M-element buckets, 10 steps: every
    rank steps its shard as one call per non-empty bucket range (the slices are
    views of the source ranks' full gradients, as a ReduceScatter output
    would be), then every rank assembles the others' slots. Every rank's
    master, m, v and slot equal the oracle's bit for bit, and every rank's full
    flat buffer is the concatenation of the oracle's slots."""
    w = GPT2_SMALL
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align,
                              bucket_elems=w.bucket_elems)
    N, S, P, P_pad = plan.world, plan.S, plan.P, plan.P_pad
    ranges = []
    for r in range(N):
        rr = [zs.zs_plan_bucket(plan, b, r) for b in range(plan.n_buckets)]
        rr = [(lo, hi) for lo, hi in rr if hi > lo]
        assert sum(hi - lo for lo, hi in rr) == S
        ranges.append(rr)
    assert max(len(rr) for rr in ranges) >= 2
    grad_kw = dict(seed=w.seed, sigma=w.grad_sigma, bf16=True)
    master_kw = dict(seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma)
    stream = torch.cuda.current_stream().cuda_stream
    d_local = [torch.empty(P_pad, dtype=torch.int16, device=DEV) for _ in range(N)]
    d_master = [dev_fill(S, bf16=False, index0=r * S, p_limit=P, **master_kw) for r in range(N)]
    d_m = [torch.zeros(S, dtype=torch.float32, device=DEV) for _ in range(N)]
    d_v = [torch.zeros(S, dtype=torch.float32, device=DEV) for _ in range(N)]
    d_full = [torch.zeros(P_pad, dtype=torch.int16, device=DEV) for _ in range(N)]
    for t in range(1, w.steps + 1):
        for j in range(N):
            synth.fill_device(d_local[j].data_ptr(), P_pad, rank=j, step=t, p_limit=P,
                              cuda_stream=stream, **grad_kw)
        for r in range(N):
            slices = [d_local[j].narrow(0, r * S, S) for j in range(N)]
            for lo, hi in ranges[r]:
                zs.zs_shard_step(plan, r, lo, hi, slices, zs.ZS_BF16, d_master[r], d_m[r], d_v[r],
                                 d_full[r], zs.ZS_BF16, w.hparams, t)
    for r in range(N):
        own = [d_full[j].narrow(0, j * S, S) for j in range(N)]
        zs.zs_gather_assemble(plan, r, own, d_full[r], zs.ZS_BF16)
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    full0 = _host(d_full[0], np.uint8)
    for r in range(1, N):
        assert np.array_equal(_host(d_full[r], np.uint8), full0), f"rank {r} assembled another buffer"
    diff = 0
    for r in range(N):
        check = bitwise_check(_host(d_master[r], np.float32), _host(d_m[r], np.float32),
                              _host(d_v[r], np.float32),
                              {oracle.BF16: full0[2 * r * S:2 * (r + 1) * S]})
        diff += oracle_chunks(orc, world=N, rank=r, S=S, P=P, steps=w.steps, hp=w.hparams,
                              grad_kw=grad_kw, master_kw=master_kw, pdts=[oracle.BF16],
                              check=check)
    assert diff == 0, f"{diff} elements differ in some bit (within the gates)"
    assert not full0[2 * P:].any(), "tail pad of the flat buffer"
    plan.free()


PDTS = [(zs.ZS_BF16, oracle.BF16), (zs.ZS_FP24, oracle.FP24), (zs.ZS_FP32, oracle.FP32)]


def _sweep_point(N, S, gb, steps, together=True):
    """The sweep's launch configuration (one tensor of N*S elements, rank 0's
    step) for every parameter dtype from the same inputs: returns host copies
    of the final master, m, v (identical for every parameter dtype, checked)
    and each dtype's slot bytes. together=False runs the parameter dtypes one
    after another (one state and one flat buffer on the device at a time, the
    slices regenerated for each)."""
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
    assert plan.S == S
    stream = torch.cuda.current_stream().cuda_stream
    bf16 = gb == 2
    gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
    grads = [torch.empty(S * gb, dtype=torch.uint8, device=DEV) for _ in range(N)]
    host_states, slots = [], {}

    def run(pdts):
        states, fulls = [], []
        for zdt, odt in pdts:
            master = torch.empty(S, dtype=torch.float32, device=DEV)
            synth.fill_device(master.data_ptr(), S, seed=1, stream=synth.STREAM_MASTER,
                              sigma=0.02, bf16=False, cuda_stream=stream)
            states.append((master, torch.zeros(S, dtype=torch.float32, device=DEV),
                           torch.zeros(S, dtype=torch.float32, device=DEV)))
            fulls.append(torch.zeros(N * S * oracle.ELEM_BYTES[odt], dtype=torch.uint8,
                                     device=DEV))
        for t in range(1, steps + 1):
            for j, g in enumerate(grads):
                synth.fill_device(g.data_ptr(), S, seed=1, rank=j, step=t, sigma=1e-3, bf16=bf16,
                                  cuda_stream=stream)
            for (zdt, odt), st, full in zip(pdts, states, fulls):
                zs.zs_shard_step(plan, 0, 0, S, grads, gdt, *st, full, zdt, HP, t)
        torch.cuda.synchronize()
        zs.zs_check_device_error()
        for (zdt, odt), st, full in zip(pdts, states, fulls):
            host_states.append(tuple(_host(x, np.float32) for x in st))
            eb = oracle.ELEM_BYTES[odt]
            assert all_zero(full[S * eb:]), "another rank's slot was written"
            slots[odt] = _host(full[:S * eb], np.uint8)
        del states, fulls
        torch.cuda.empty_cache()

    if together:
        run(PDTS)
    else:
        for p in PDTS:
            run([p])
    for hs in host_states[1:]:
        for a, b in zip(hs, host_states[0]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    del grads
    torch.cuda.empty_cache()
    plan.free()
    return host_states[0], slots


@pytest.mark.parametrize("gb", [2, 4], ids=["bf16_slices", "fp32_slices"])
@pytest.mark.parametrize("N", SWEEP_WORLDS)
@pytest.mark.parametrize("log2S", [22, 24])
def test_sweep_every_element(orc, log2S, N, gb):
    """Sweep grid at S = 2^22 and 2^24 (the sizes where the per-call kernel
    choice and the staged kernel's launch shape change with N and the dtypes),
    3 steps, bf16 / 3-byte / fp32 parameters: every element bit for bit."""
    S, steps = 1 << log2S, 3
    (g_master, g_m, g_v), slots = _sweep_point(N, S, gb, steps)
    check = bitwise_check(g_master, g_m, g_v, slots)
    diff = oracle_chunks(orc, world=N, rank=0, S=S, P=S, steps=steps, hp=HP,
                         grad_kw=dict(seed=1, sigma=1e-3, bf16=gb == 2),
                         master_kw=dict(seed=1, stream=synth.STREAM_MASTER, sigma=0.02),
                         pdts=[p[1] for p in PDTS], check=check)
    assert diff == 0, f"{diff} elements differ in some bit (within the gates)"


@pytest.mark.parametrize("gb", [2, 4], ids=["bf16_slices", "fp32_slices"])
@pytest.mark.parametrize("N", SWEEP_WORLDS)
def test_sweep_sampled_2p28(orc, N, gb):
    """Sweep grid at S = 2^28, 2 steps, bf16 / 3-byte / fp32 parameters:
    60,000 sampled elements, both ends of the shard and a run across a tile
    boundary, recomputed by the oracle from the regenerated inputs."""
    S, steps = 1 << 28, 2
    need = N * S * gb + 12 * S + N * S * 4
    if need > 0.8 * torch.cuda.mem_get_info()[0]:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory")
    (g_master, g_m, g_v), slots = _sweep_point(N, S, gb, steps, together=False)
    rng = np.random.default_rng(N * 10 + gb)
    idx = np.unique(np.concatenate([rng.integers(0, S, size=60_000), np.arange(0, 64),
                                    np.arange(S - 64, S),
                                    np.arange((S >> 1) - 2048, (S >> 1) + 2048)]))
    K = idx.size
    o_master = synth.at(idx, seed=1, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=S)
    o_m, o_v = np.zeros(K, np.float32), np.zeros(K, np.float32)
    bf16 = gb == 2
    for t in range(1, steps + 1):
        g_host = [synth.at(idx, seed=1, rank=j, step=t, sigma=1e-3, bf16=bf16, p_limit=S)
                  for j in range(N)]
        if t < steps:
            orc.shard_step(world=N, rank=0, S=K, lo=0, hi=K, grads=g_host, master=o_master,
                           m=o_m, v=o_v, full_flat=np.zeros(4 * K, np.uint8), t=t, **oracle_hp(HP))
            continue
        for _, odt in PDTS:
            st = [o_master.copy(), o_m.copy(), o_v.copy()]
            eb = oracle.ELEM_BYTES[odt]
            out = np.zeros(K * eb, np.uint8)
            orc.shard_step(world=N, rank=0, S=K, lo=0, hi=K, grads=g_host, master=st[0], m=st[1],
                           v=st[2], full_flat=out, param_dtype=odt, t=t, **oracle_hp(HP))
            bi = (idx[:, None] * eb + np.arange(eb)[None, :]).reshape(-1)
            assert np.array_equal(slots[odt][bi], out), odt
            assert assert_params_close(slots[odt][bi], out, odt) == 0
        o_master, o_m, o_v = st
    for name, got, ref in (("master", g_master, o_master), ("m", g_m, o_m), ("v", g_v, o_v)):
        assert assert_state_close(got[idx], ref, name) == 0
        assert np.array_equal(got[idx].view(np.uint32), ref.view(np.uint32)), name


def test_qwen25_3b_accumulated_clipped_every_element(orc):
    """Gradient accumulation with clipping at full size (Qwen2.5-3B, N = 4,
    rank 1, 771,484,672 elements): G = 2 micro-batches per optimizer step, two
    optimizer steps; each step accumulates the first micro-batch's mean, takes
    the norm of the accumulated step's gradient, forms the clip coefficient
    from the N ranks' partial sums (every rank's taken equal to this one's, the
    emulated AllReduce) with max_norm at half the norm so that the step clips,
    and runs the clipped accumulated step. The oracle, chunk by chunk over the
    whole shard, runs the same micro-steps with the coefficient the device
    formed (the coefficient from given partials is compared bit for bit in
    test_gpu_clip.py); master, m, v and the slot bit for bit; each step's norm
    against the oracle's sequential sum within that sum's rounding bound."""
    w, rank, G, T = QWEN25_3B, 1, 2, 2
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    grad_kw = dict(seed=w.seed, sigma=w.grad_sigma, bf16=True)
    master_kw = dict(seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma)
    stream = torch.cuda.current_stream().cuda_stream
    d_master = dev_fill(S, bf16=False, index0=rank * S, p_limit=P, **master_kw)
    d_m = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_v = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    d_acc = torch.empty(S, dtype=torch.float32, device=DEV)
    d_grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)
    parts = torch.zeros(N, dtype=torch.float64, device=DEV)
    coef = torch.zeros(1, dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    coefs, norms = [], []
    for t in range(1, T + 1):
        for mstep in range(1, G + 1):
            for j in range(N):
                synth.fill_device(d_grads[j].data_ptr(), S, index0=rank * S, rank=j,
                                  step=(t - 1) * G + mstep, p_limit=P, cuda_stream=stream,
                                  **grad_kw)
            if mstep < G:
                zs.zs_grad_accumulate(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_acc, mstep == 1)
                continue
            zs.zs_grad_sqnorm_accumulated(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_acc, G, ws,
                                          parts.narrow(0, rank, 1))
            torch.cuda.synchronize()
            own = float(parts[rank].item())
            parts.fill_(own)
            norms.append(own)
            zs.zs_clip_coefficient(parts, N, 0.5 * (N * own) ** 0.5, coef, bad)
            zs.zs_shard_step_accumulated_clipped(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_acc, G,
                                                 d_master, d_m, d_v, d_full, zs.ZS_BF16,
                                                 w.hparams, t, coef, bad)
            torch.cuda.synchronize()
            coefs.append(float(coef.item()))
            assert int(bad.item()) == 0 and 0.0 < coefs[-1] < 1.0
    zs.zs_check_device_error()
    del d_grads, d_acc
    g_master, g_m, g_v = _host(d_master, np.float32), _host(d_m, np.float32), _host(d_v, np.float32)
    g_slot = _host(d_full.narrow(0, rank * S, S), np.uint8)
    del d_master, d_m, d_v, d_full
    torch.cuda.empty_cache()
    check = bitwise_check(g_master, g_m, g_v, {oracle.BF16: g_slot})
    hpo = oracle_hp(w.hparams)
    sq = np.zeros((S + CHUNK - 1) // CHUNK * T).reshape(-1, T)

    def work(c0, c1):
        n = c1 - c0
        master = synth.fill(n, index0=rank * S + c0, p_limit=P, threads=1, **master_kw)
        m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
        acc = np.zeros(n, np.float32)
        slot = np.zeros(n * 2, np.uint8)
        for t in range(1, T + 1):
            for mstep in range(1, G + 1):
                grads = [synth.fill(n, index0=rank * S + c0, rank=j, step=(t - 1) * G + mstep,
                                    p_limit=P, threads=1, **grad_kw) for j in range(N)]
                if mstep < G:
                    orc.grad_accumulate(world=N, S=n, lo=0, hi=n, grads=grads, accum=acc,
                                        first=mstep == 1)
                    continue
                sq[c0 // CHUNK, t - 1] = orc.grad_sqnorm_accumulated(
                    world=N, S=n, lo=0, hi=n, grads=grads, accum=acc, micro_steps=G)
                orc.shard_step_accumulated_clipped(
                    world=N, rank=0, S=n, lo=0, hi=n, grads=grads, accum=acc, micro_steps=G,
                    master=master, m=m, v=v, full_flat=slot, coef=np.float32(coefs[t - 1]),
                    skip=0, t=t, **hpo)
        return check(c0, c1, master, m, v, {oracle.BF16: slot})

    diff = run_chunks(work, 0, S)
    assert diff == 0, f"{diff} elements differ in some bit (within the gates)"
    for t in range(T):
        want = float(np.sum(sq[:, t]))   # chunk sums added in chunk order
        assert abs(norms[t] - want) <= (S + 16) * 2.0 ** -52 * want, (t, norms[t], want)
    plan.free()


def test_qwen25_3b_every_wrap_unit_copy_out(orc):
    """FSDP2's copy-out at full size in the benchmark's launch configuration:
    every wrap unit of Qwen2.5-3B (36 blocks + the root unit with the tied
    embedding, N = 4, rows sharded per parameter), the rank-major gathered
    buffer from the generator, one zs_unshard per unit; every parameter element
    against the oracle's copy-out of the same gathered bytes."""
    from synth.workloads import wrap_units
    w = QWEN25_3B
    stream = torch.cuda.current_stream().cuda_stream
    units = wrap_units(w)
    assert len(units) == 37
    for k, idx in enumerate(units):
        local_of = {g: i for i, g in enumerate(idx)}
        ps = [w.params[i] for i in idx]
        ties = [local_of[p.tied_to] if p.tied_to >= 0 else -1 for p in ps]
        dims, numels = [p.shape[0] for p in ps], [p.numel for p in ps]
        plan = zs.zs_rows_plan(dims, numels, ties, world=w.world, align_elems=w.align)
        rp = orc.rows_plan(dims, numels, ties, world=w.world, align=w.align)
        assert plan.P_pad == w.world * rp["S"]
        gbuf = torch.empty(plan.P_pad, dtype=torch.int16, device=DEV)
        synth.fill_device(gbuf.data_ptr(), plan.P_pad, seed=w.seed, rank=k, step=1,
                          sigma=w.grad_sigma, bf16=True, cuda_stream=stream)
        outs = [torch.empty(n, dtype=torch.int16, device=DEV) if t < 0 else None
                for n, t in zip(numels, ties)]
        zs.zs_unshard(plan, gbuf, zs.ZS_BF16, outs)
        g_host = synth.fill(plan.P_pad, seed=w.seed, rank=k, step=1, sigma=w.grad_sigma,
                            bf16=True)
        refs = [np.zeros(n, np.uint16) if t < 0 else None for n, t in zip(numels, ties)]
        orc.unshard(rp, g_host.view(np.uint8), 2,
                    [None if x is None else x.view(np.uint8) for x in refs])
        torch.cuda.synchronize()
        for i, (d, r) in enumerate(zip(outs, refs)):
            if r is not None:
                assert np.array_equal(_host(d, np.uint16), r), (k, ps[i].name)
        del gbuf, outs
        plan.free()
    zs.zs_check_device_error()
    torch.cuda.empty_cache()


def test_llama_7b_gather_every_element(orc):
    """The emulated AllGather's assembly at full size (Llama-7B, N = 8, rank 5's
    view): the other seven ranks' bf16 shards (842M elements each) into the
    13.5 GB flat buffer, in the benchmark's launch configuration; every byte
    against the oracle's gather of the same shards, the own slot untouched."""
    w, rank = LLAMA_7B, 5
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P_pad = plan.world, plan.S, plan.P_pad
    stream = torch.cuda.current_stream().cuda_stream
    kw = dict(seed=w.seed, step=3, sigma=w.grad_sigma, bf16=True)
    srcs = []
    for j in range(N):
        if j == rank:
            srcs.append(None)
            continue
        t = torch.empty(S, dtype=torch.int16, device=DEV)
        synth.fill_device(t.data_ptr(), S, index0=j * S, rank=j, cuda_stream=stream, **kw)
        srcs.append(t)
    full = torch.full((P_pad,), 0x1234, dtype=torch.int16, device=DEV)
    views = zs.zs_gather_assemble(plan, rank, srcs, full, zs.ZS_BF16)
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    del srcs
    got = _host(full, np.uint16)
    del full
    torch.cuda.empty_cache()
    expect = np.full(P_pad, 0x1234, np.uint16)
    shards = [None if j == rank else synth.fill(S, index0=j * S, rank=j, **kw)
              for j in range(N)]
    orc.gather(world=N, S=S, elem_size=2, shards=shards, full_flat=expect)
    assert np.array_equal(got, expect)
    offs = zs.zs_plan_offsets(plan)
    assert [v - views[0] for v in views] == [2 * (o - offs[0]) for o in offs]
    plan.free()


def test_llama_7b_resume_into_half_world(orc, tmp_path):
    """The pages' resume criterion at full size ("从 Data Parallel 到 ZeRO/FSDP",
    "Checkpoint 不能假设每个 Rank 都有完整模型": verify that the next update
    equals the uninterrupted run): Llama-7B at N = 8, ranks 0 and 1 take a
    step and save their fp32 master / m / v (10.1 GB each); rank 0 of the same
    model at N = 4 restores from those two files. The restored shard is the two
    old shards back to back, bit for bit; then the next step, with every
    rank's gradient equal to one bf16 x (its mean is x at any power-of-two
    world), leaves the restored rank's master, m, v and parameters equal to the
    uninterrupted ranks' bit for bit."""
    w = LLAMA_7B
    pa = zs.zs_flatten_plan(w.numels, w.tied_to, world=8, align_elems=w.align)
    pb = zs.zs_flatten_plan(w.numels, w.tied_to, world=4, align_elems=w.align)
    S, Sb, P = pa.S, pb.S, pa.P
    assert Sb == 2 * S and pa.P_pad == pb.P_pad
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(8)]
    full_a = torch.zeros(pa.P_pad, dtype=torch.int16, device=DEV)
    state, paths = [], []
    for r in (0, 1):
        st = (dev_fill(S, bf16=False, index0=r * S, seed=w.seed, stream=synth.STREAM_MASTER,
                       sigma=w.master_sigma, p_limit=P),
              torch.zeros(S, dtype=torch.float32, device=DEV),
              torch.zeros(S, dtype=torch.float32, device=DEV))
        for j in range(8):
            synth.fill_device(grads[j].data_ptr(), S, index0=r * S, seed=w.seed, rank=j, step=1,
                              sigma=w.grad_sigma, p_limit=P, outlier_frac=w.outlier_frac,
                              outlier_scale=w.outlier_scale, bf16=True, cuda_stream=stream)
        zs.zs_shard_step(pa, r, 0, S, grads, zs.ZS_BF16, *st, full_a, zs.ZS_BF16, w.hparams, 1)
        paths.append(str(tmp_path / f"llama7b.rank{r}"))
        zs.zs_checkpoint_save(pa, r, *st, 1, paths[-1])
        state.append(st)
    del grads
    torch.cuda.empty_cache()
    restored = [torch.empty(Sb, dtype=torch.float32, device=DEV) for _ in range(3)]
    assert zs.zs_checkpoint_load(pb, 0, paths + [None] * 6, *restored) == 1
    for k in range(3):
        assert torch.equal(restored[k].view(torch.int32),
                           torch.cat([state[0][k], state[1][k]]).view(torch.int32)), k
    for p in paths:
        os.remove(p)
    # the next update, uninterrupted (N = 8, ranks 0 and 1) and restored (N = 4, rank 0)
    x = torch.empty(Sb, dtype=torch.int16, device=DEV)
    synth.fill_device(x.data_ptr(), Sb, seed=77, step=2, sigma=w.grad_sigma, p_limit=P,
                      bf16=True, cuda_stream=stream)
    for r in (0, 1):
        xr = x.narrow(0, r * S, S)
        zs.zs_shard_step(pa, r, 0, S, [xr] * 8, zs.ZS_BF16, *state[r], full_a, zs.ZS_BF16,
                         w.hparams, 2)
    full_b = torch.zeros(pb.P_pad, dtype=torch.int16, device=DEV)
    zs.zs_shard_step(pb, 0, 0, Sb, [x] * 4, zs.ZS_BF16, *restored, full_b, zs.ZS_BF16,
                     w.hparams, 2)
    torch.cuda.synchronize()
    zs.zs_check_device_error()
    for k in range(3):
        assert torch.equal(restored[k].view(torch.int32),
                           torch.cat([state[0][k], state[1][k]]).view(torch.int32)), k
    assert torch.equal(full_b[:Sb], full_a[:Sb])
    pa.free()
    pb.free()
