"""GPU parity of gradient accumulation on the shard: G micro-steps through
zs_grad_accumulate and zs_shard_step_accumulated against the oracle's same
pipeline, element by element (fp32 state within 1e-6 relative and, as the
operations are the same IEEE ones, bit for bit; parameters within 1 ulp)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import (DEV, ZS_OF, assert_params_close, assert_state_close, dev_fill,
                      oracle_hp, to_dev, to_host)
from synth.workloads import GPT2_SMALL

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _buf(nbytes, fill, front):
    whole = torch.zeros(front + nbytes + 64, dtype=torch.uint8, device=DEV)
    inner = whole.narrow(0, front, nbytes)
    inner.copy_(torch.from_numpy(np.ascontiguousarray(fill).view(np.uint8)).to(DEV))
    return inner


@pytest.mark.parametrize("seed", range(12))
def test_random_accumulation_cases(orc, seed):
    rng = np.random.default_rng(500 + seed)
    N = int(rng.choice([1, 2, 4, 8, 16]))
    G = int(rng.integers(1, 5))
    S0 = int(rng.integers(1, 20000))
    align = int(rng.choice([128, 1]))
    plan = zs.zs_flatten_plan([N * S0 - int(rng.integers(0, 7))], world=N, align_elems=align)
    S, P = plan.S, plan.P
    rank = int(rng.integers(0, N))
    lo = int(rng.integers(0, S // 4 + 1))
    hi = int(rng.integers(max(lo, 3 * S // 4), S + 1))
    bf16 = seed % 3 != 2
    pdt = int(rng.choice([oracle.BF16, oracle.BF16, oracle.FP24, oracle.FP32]))
    eb = oracle.ELEM_BYTES[pdt]
    front = 16 if seed % 4 == 1 else 0
    master0 = synth.fill(S, index0=rank * S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02,
                         p_limit=P)
    o_st = [master0.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    o_acc = np.zeros(S, np.float32)
    o_full = np.zeros(plan.P_pad * eb, np.uint8)
    d_st = [_buf(S * 4, x, front) for x in o_st]
    d_acc = _buf(S * 4, np.full(S, np.nan, np.float32), front)   # stale contents
    d_full = _buf(plan.P_pad * eb, o_full, 0)
    gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
    for t in (1, 2):
        for k in range(G):
            host = [synth.fill(S, index0=rank * S, seed=seed, rank=j, step=10 * t + k, p_limit=P,
                               bf16=bf16) for j in range(N)]
            dev = [_buf(h.nbytes, h, front) for h in host]
            if k < G - 1:
                zs.zs_grad_accumulate(plan, rank, lo, hi, dev, gdt, d_acc, k == 0)
                orc.grad_accumulate(world=N, S=S, lo=lo, hi=hi, grads=host, accum=o_acc,
                                    first=k == 0)
            else:
                if G == 1:
                    d_acc.zero_()
                    o_acc[:] = 0
                zs.zs_shard_step_accumulated(plan, rank, lo, hi, dev, gdt, d_acc, G, *d_st,
                                             d_full, ZS_OF[pdt], HP, t)
                orc.shard_step_accumulated(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=host,
                                           accum=o_acc, micro_steps=G, master=o_st[0],
                                           m=o_st[1], v=o_st[2], full_flat=o_full,
                                           param_dtype=pdt, t=t, **oracle_hp(HP))
        torch.cuda.synchronize()
        if G > 1:
            got_acc = to_host(d_acc, np.float32)[lo:hi]
            assert assert_state_close(got_acc, o_acc[lo:hi], "accum") == 0
        for name, d, ref in zip(("master", "m", "v"), d_st, o_st):
            assert assert_state_close(to_host(d, np.float32), ref, name) == 0
        got = to_host(d_full, np.uint8)
        assert assert_params_close(got, o_full, pdt) == 0
        assert np.array_equal(got, o_full)
    plan.free()


def test_gpt2_small_accumulation_full_size(orc):
    """GPT-2-small list, N = 8, rank 6, G = 4 micro-steps, 2 optimizer steps:
    every element of the shard against the oracle."""
    w = GPT2_SMALL
    G, rank = 4, 6
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    hp = w.hparams
    d_master = dev_fill(S, bf16=False, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                        sigma=w.master_sigma, p_limit=P)
    d_m = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_v = torch.zeros(S, dtype=torch.float32, device=DEV)
    d_acc = torch.empty(S, dtype=torch.float32, device=DEV)
    d_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    o_master = synth.fill(S, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                          sigma=w.master_sigma, p_limit=P)
    o_m, o_v = np.zeros(S, np.float32), np.zeros(S, np.float32)
    o_acc = np.zeros(S, np.float32)
    o_full = np.zeros(plan.P_pad, np.uint16)
    d_grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    for t in (1, 2):
        for k in range(G):
            key = dict(index0=rank * S, seed=w.seed, step=100 * t + k, sigma=w.grad_sigma,
                       p_limit=P, bf16=True)
            for j in range(N):
                synth.fill_device(d_grads[j].data_ptr(), S, rank=j,
                                  cuda_stream=torch.cuda.current_stream().cuda_stream, **key)
            host = [synth.fill(S, rank=j, **key) for j in range(N)]
            if k < G - 1:
                zs.zs_grad_accumulate(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_acc, k == 0)
                orc.grad_accumulate(world=N, S=S, lo=0, hi=S, grads=host, accum=o_acc,
                                    first=k == 0)
            else:
                zs.zs_shard_step_accumulated(plan, rank, 0, S, d_grads, zs.ZS_BF16, d_acc, G,
                                             d_master, d_m, d_v, d_full, zs.ZS_BF16, hp, t)
                orc.shard_step_accumulated(world=N, rank=rank, S=S, lo=0, hi=S, grads=host,
                                           accum=o_acc, micro_steps=G, master=o_master, m=o_m,
                                           v=o_v, full_flat=o_full, t=t, **oracle_hp(hp))
    torch.cuda.synchronize()
    for name, d, ref in (("master", d_master, o_master), ("m", d_m, o_m), ("v", d_v, o_v)):
        assert assert_state_close(to_host(d, np.float32), ref, name) == 0
    got = to_host(d_full, np.uint16)
    assert assert_params_close(got, o_full, oracle.BF16) == 0
    assert np.array_equal(got, o_full)
    plan.free()


def test_accumulation_argument_errors():
    plan = zs.zs_flatten_plan([4096], world=4)
    S = plan.S
    g = [torch.zeros(S, dtype=torch.int16, device=DEV) for _ in range(4)]
    st = [torch.zeros(S, device=DEV) for _ in range(4)]
    full = torch.zeros(4096, dtype=torch.int16, device=DEV)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_shard_step_accumulated(plan, 0, 0, S, g, zs.ZS_BF16, st[3], 0, *st[:3], full,
                                     zs.ZS_BF16, HP, 1)
    assert e.value.status == zs.ZS_ERR_RANGE
    with pytest.raises(zs.ZsError) as e:   # accumulator aliasing the master
        zs.zs_shard_step_accumulated(plan, 0, 0, S, g, zs.ZS_BF16, st[0], 2, *st[:3], full,
                                     zs.ZS_BF16, HP, 1)
    assert e.value.status == zs.ZS_ERR_INVAL
    with pytest.raises(zs.ZsError) as e:   # accumulator aliasing a slice
        zs.zs_grad_accumulate(plan, 0, 0, S, g, zs.ZS_BF16, g[1].data_ptr(), True)
    assert e.value.status == zs.ZS_ERR_INVAL
    plan.free()
