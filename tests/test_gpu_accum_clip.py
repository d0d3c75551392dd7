"""GPU parity of clipping an accumulated gradient: the norm pass over the
accumulated step's gradient ((accum + mean) * 1/G) against the oracle's
sequential sum (within that sum's rounding bound, the same on every run); the
clipped accumulated step bit for bit against the oracle given the oracle's own
coefficient, on both step kernels; the whole pipeline (G micro-steps on N
ranks, the partial norms, the coefficient, the clipped steps) against the
oracle's pipeline, including a NaN that makes every rank skip; and the new
entry points' argument checks."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import (DEV, ZS_OF, assert_params_close, assert_state_close, oracle_hp, to_dev,
                      to_host)

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def sum_bound(n):
    """Relative rounding bound of the oracle's sequential double sum of n
    non-negative terms, with room for the GPU's own, much smaller, error."""
    return (n + 16) * 2.0 ** -52


def _buf(nbytes, fill, front):
    whole = torch.zeros(front + nbytes + 64, dtype=torch.uint8, device=DEV)
    inner = whole.narrow(0, front, nbytes)
    inner.copy_(torch.from_numpy(np.ascontiguousarray(fill).view(np.uint8)).to(DEV))
    return inner


def workspace():
    return torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("seed", range(10))
def test_accumulated_norm_random_cases(orc, seed):
    rng = np.random.default_rng(900 + seed)
    N = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    G = int(rng.integers(1, 6))
    S0 = int(rng.integers(1, 30000)) if seed % 3 else int(rng.integers(1, 40)) * 16
    plan = zs.zs_flatten_plan([N * S0], world=N, align_elems=1)
    S = plan.S
    bf16 = seed % 4 != 3
    front = 16 if seed % 5 == 2 else 0          # 16-byte aligned only: element path
    host = [synth.fill(S, seed=seed, rank=j, step=1, bf16=bf16, outlier_frac=0.01,
                       outlier_scale=100.0) for j in range(N)]
    acc = (rng.standard_normal(S) * 3e-3).astype(np.float32)
    dev = [_buf(h.nbytes, h, front) for h in host]
    d_acc = _buf(S * 4, acc, front)
    lo = int(rng.integers(0, S // 3 + 1))
    hi = int(rng.integers(max(lo, 2 * S // 3), S + 1))
    gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
    ws = workspace()
    out = [torch.zeros(1, dtype=torch.float64, device=DEV) for _ in range(2)]
    for o in out:
        zs.zs_grad_sqnorm_accumulated(plan, 0, lo, hi, dev, gdt, d_acc, G, ws, o)
    ref = orc.grad_sqnorm_accumulated(world=N, S=S, lo=lo, hi=hi, grads=host, accum=acc,
                                      micro_steps=G)
    got = float(out[0].item())
    assert float(out[1].item()) == got, "norm pass is not reproducible"
    assert abs(got - ref) <= sum_bound(hi - lo) * ref + 1e-300, (got, ref)
    plan.free()


@pytest.mark.parametrize("path", [zs.STEP_PATH_DIRECT, zs.STEP_PATH_STAGED])
@pytest.mark.parametrize("pdt", [oracle.BF16, oracle.FP24])
def test_accumulated_clipped_step_bit_exact(orc, path, pdt):
    """Given the oracle's coefficient (written to the device), the GPU's
    clipped accumulated step equals the oracle's bit for bit, over a ragged
    sub-range, on the register-streaming and the staged kernel."""
    N, G, S0 = 4, 3, 41_000
    plan = zs.zs_flatten_plan([N * S0], world=N, align_elems=128)
    S, rank = plan.S, 2
    lo, hi = 37, S - 11
    eb = oracle.ELEM_BYTES[pdt]
    host = [synth.fill(S, seed=7, rank=j, step=3, bf16=True) for j in range(N)]
    acc = (np.random.default_rng(8).standard_normal(S) * 2e-3).astype(np.float32)
    master0 = synth.fill(S, seed=7, stream=synth.STREAM_MASTER, sigma=0.02)
    o_st = [master0.copy(), np.full(S, 1e-4, np.float32), np.full(S, 1e-7, np.float32)]
    o_full = np.zeros(plan.P_pad * eb, np.uint8)
    sq = orc.grad_sqnorm_accumulated(world=N, S=S, lo=0, hi=S, grads=host, accum=acc,
                                     micro_steps=G)
    coef, bad = orc.clip_coef([sq], 0.4 * float(np.sqrt(sq)))
    assert bad == 0 and coef < 1
    d_st = [to_dev(x.copy()) for x in o_st]
    d_full = torch.zeros(plan.P_pad * eb, dtype=torch.uint8, device=DEV)
    d_coef = torch.tensor([coef], dtype=torch.float32, device=DEV)
    d_skip = torch.zeros(1, dtype=torch.int32, device=DEV)
    old = zs.zs_set_step_path(path)
    try:
        zs.zs_shard_step_accumulated_clipped(plan, rank, lo, hi, [to_dev(h) for h in host],
                                             zs.ZS_BF16, to_dev(acc), G, *d_st, d_full,
                                             ZS_OF[pdt], HP, 5, coef=d_coef, skip=d_skip)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_step_path(old)
    orc.shard_step_accumulated_clipped(world=N, rank=rank, S=S, lo=lo, hi=hi, grads=host,
                                       accum=acc, micro_steps=G, master=o_st[0], m=o_st[1],
                                       v=o_st[2], full_flat=o_full, coef=coef, skip=0,
                                       param_dtype=pdt, t=5, **oracle_hp(HP))
    for name, d, ref in zip(("master", "m", "v"), d_st, o_st):
        got = to_host(d, np.float32)
        assert assert_state_close(got, ref, name) == 0
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), name
    got = to_host(d_full, np.uint8)
    assert assert_params_close(got, o_full, pdt) == 0
    assert np.array_equal(got, o_full)
    plan.free()


def _pipeline(orc, N, S0, G, seed, max_norm_frac, poison=None, steps=2):
    plan = zs.zs_flatten_plan([N * S0], world=N)
    S = plan.S
    master0 = synth.fill(S * N, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02)
    o_st = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
            for r in range(N)]
    o_acc = [np.zeros(S, np.float32) for _ in range(N)]
    o_full = [np.zeros(S * N, np.uint16) for _ in range(N)]
    d_st = [[to_dev(x.copy()) for x in st] for st in o_st]
    d_acc = [torch.full((S,), float("nan"), dtype=torch.float32, device=DEV) for _ in range(N)]
    d_full = [torch.zeros(S * N, dtype=torch.int16, device=DEV) for _ in range(N)]
    ws = workspace()
    parts = torch.zeros(N, dtype=torch.float64, device=DEV)
    coef = torch.zeros(1, dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    max_norm = None
    seen = []
    for t in range(1, steps + 1):
        for k in range(G):
            local = [synth.fill(S * N, seed=seed, rank=j, step=100 * t + k, bf16=True)
                     for j in range(N)]
            if poison is not None and t == steps and k == G - 1:
                local[poison[0]][poison[1]] = 0x7FC0
            slices = [[local[j][r * S:(r + 1) * S].copy() for j in range(N)] for r in range(N)]
            d_slices = [[to_dev(x) for x in sl] for sl in slices]
            if k < G - 1:
                for r in range(N):
                    orc.grad_accumulate(world=N, S=S, lo=0, hi=S, grads=slices[r],
                                        accum=o_acc[r], first=k == 0)
                    zs.zs_grad_accumulate(plan, r, 0, S, d_slices[r], zs.ZS_BF16, d_acc[r],
                                          k == 0)
                continue
            o_parts = [orc.grad_sqnorm_accumulated(world=N, S=S, lo=0, hi=S, grads=slices[r],
                                                   accum=o_acc[r], micro_steps=G)
                       for r in range(N)]
            if max_norm is None:
                max_norm = max_norm_frac * float(np.sqrt(sum(o_parts)))
            o_coef, o_bad = orc.clip_coef(o_parts, max_norm)
            for r in range(N):
                orc.shard_step_accumulated_clipped(world=N, rank=r, S=S, lo=0, hi=S,
                                                   grads=slices[r], accum=o_acc[r],
                                                   micro_steps=G, master=o_st[r][0],
                                                   m=o_st[r][1], v=o_st[r][2],
                                                   full_flat=o_full[r], coef=o_coef,
                                                   skip=o_bad, t=t, **oracle_hp(HP))
            for r in range(N):
                zs.zs_grad_sqnorm_accumulated(plan, r, 0, S, d_slices[r], zs.ZS_BF16, d_acc[r],
                                              G, ws, parts.narrow(0, r, 1))
            zs.zs_clip_coefficient(parts, N, max_norm, coef, bad)
            for r in range(N):
                zs.zs_shard_step_accumulated_clipped(plan, r, 0, S, d_slices[r], zs.ZS_BF16,
                                                     d_acc[r], G, *d_st[r], d_full[r],
                                                     zs.ZS_BF16, HP, t, coef=coef, skip=bad)
            torch.cuda.synchronize()
            seen.append((float(coef.item()), int(bad.item()), float(o_coef), o_bad))
            assert int(bad.item()) == o_bad
            g_parts = parts.cpu().numpy()
            for r in range(N):
                if np.isfinite(o_parts[r]):
                    assert abs(g_parts[r] - o_parts[r]) <= sum_bound(S) * o_parts[r]
    for r in range(N):
        for name, d, ref in zip(("master", "m", "v"), d_st[r], o_st[r]):
            assert assert_state_close(to_host(d, np.float32), ref, f"{name}[{r}]") == 0
        assert assert_params_close(to_host(d_full[r], np.uint16), o_full[r], oracle.BF16) == 0
    plan.free()
    return seen


def test_accumulated_clip_pipeline_matches_oracle(orc):
    """N = 4 ranks, G = 3 micro-steps, two optimizer steps that clip
    (max_norm = 0.3 x the first accumulated norm)."""
    seen = _pipeline(orc, N=4, S0=30_000, G=3, seed=11, max_norm_frac=0.3)
    for c_gpu, bad_gpu, c_ref, bad_ref in seen:
        assert bad_gpu == bad_ref == 0 and c_gpu < 1
        assert abs(c_gpu - c_ref) <= 2 * np.spacing(np.float32(c_ref))


def test_accumulated_nonfinite_skips_every_rank(orc):
    """A NaN in one source rank's last micro-step makes the accumulated norm
    non-finite; every rank's second step leaves its buffers untouched."""
    seen = _pipeline(orc, N=4, S0=8192, G=2, seed=13, max_norm_frac=10.0, poison=(1, 4321))
    assert seen[0][1] == 0 and seen[1][1] == 1


def test_accumulated_clip_argument_errors():
    plan = zs.zs_flatten_plan([4096], world=4)
    S = plan.S
    g = [torch.zeros(S, dtype=torch.int16, device=DEV) for _ in range(4)]
    acc = torch.zeros(S, dtype=torch.float32, device=DEV)
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    ws = workspace()
    st = [torch.zeros(S, dtype=torch.float32, device=DEV) for _ in range(3)]
    full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    coef = torch.zeros(2, dtype=torch.float32, device=DEV)
    cases = [
        (lambda: zs.zs_grad_sqnorm_accumulated(plan, 0, 0, S, g, zs.ZS_BF16, acc, 0, ws, out),
         zs.ZS_ERR_RANGE),
        (lambda: zs.zs_grad_sqnorm_accumulated(plan, 0, 0, S, g, zs.ZS_BF16, None, 2, ws, out),
         zs.ZS_ERR_INVAL),
        (lambda: zs.zs_grad_sqnorm_accumulated(plan, 0, 0, S, g, zs.ZS_BF16,
                                               acc.data_ptr() + 4, 2, ws, out), zs.ZS_ERR_ALIGN),
        (lambda: zs.zs_shard_step_accumulated_clipped(plan, 0, 0, S, g, zs.ZS_BF16, acc, 0, *st,
                                                      full, zs.ZS_BF16, HP, 1), zs.ZS_ERR_RANGE),
        (lambda: zs.zs_shard_step_accumulated_clipped(plan, 0, 0, S, g, zs.ZS_BF16, None, 2, *st,
                                                      full, zs.ZS_BF16, HP, 1), zs.ZS_ERR_INVAL),
        (lambda: zs.zs_shard_step_accumulated_clipped(plan, 0, 0, S, g, zs.ZS_BF16, acc, 2, *st,
                                                      full, zs.ZS_BF16, HP, 1,
                                                      coef=coef.data_ptr() + 2), zs.ZS_ERR_ALIGN),
    ]
    for call, status in cases:
        with pytest.raises(zs.ZsError) as e:
            call()
        assert e.value.status == status, str(e.value)
    plan.free()
