"""GPU parity of global-norm clipping: the norm pass against the oracle's
sequential sum (within the sum's rounding bound; the GPU result is the same
on every run), the coefficient kernel bit for bit on the same partial sums,
the whole clipped step pipeline against the oracle's pipeline, and the shared
skip on a non-finite norm."""
import threading

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import DEV, assert_params_close, assert_state_close, oracle_hp, to_dev, to_host
from synth.workloads import GPT2_SMALL, LLAMA_7B

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def workspace():
    return torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)


def sum_bound(n):
    """Relative rounding bound of a sequential double sum of n non-negative
    terms (the oracle's), with room for the GPU's own, much smaller, error."""
    return (n + 16) * 2.0 ** -52


def gpu_sqnorm(plan, rank, lo, hi, slices, gdt, ws=None):
    ws = workspace() if ws is None else ws
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    zs.zs_grad_sqnorm(plan, rank, lo, hi, slices, gdt, ws, out)
    return out


@pytest.mark.parametrize("seed", range(10))
def test_sqnorm_random_cases(orc, seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    S = int(rng.integers(1, 40000)) if seed % 3 else int(rng.integers(1, 40)) * 16
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=1)
    S = plan.S
    bf16 = seed % 4 != 3
    host = [synth.fill(S, seed=seed, rank=j, step=1, bf16=bf16, outlier_frac=0.01,
                       outlier_scale=100.0) for j in range(N)]
    # Some cases place the slices only 16-byte aligned (element-by-element path).
    front = 16 if seed % 5 == 2 else 0
    dev = []
    for h in host:
        buf = torch.zeros(h.nbytes + 64, dtype=torch.uint8, device=DEV)
        view = buf.narrow(0, front, h.nbytes)
        view.copy_(torch.from_numpy(h.view(np.uint8)).to(DEV))
        dev.append(view)
    lo = int(rng.integers(0, S // 3 + 1))
    hi = int(rng.integers(max(lo, 2 * S // 3), S + 1))
    gdt = zs.ZS_BF16 if bf16 else zs.ZS_FP32
    a = gpu_sqnorm(plan, 0, lo, hi, dev, gdt)
    b = gpu_sqnorm(plan, 0, lo, hi, dev, gdt)
    ref = orc.grad_sqnorm(world=N, S=S, lo=lo, hi=hi, grads=host)
    got = float(a.item())
    assert float(b.item()) == got, "norm pass is not reproducible"
    assert abs(got - ref) <= sum_bound(hi - lo) * ref + 1e-300, (got, ref)
    plan.free()


def test_clip_coefficient_bit_exact_on_same_partials(orc):
    cases = [[9.0, 16.0], [4.0, 0.0, 0.0], [0.0], [1e300, 1e300], [float("inf"), 1.0],
             [1.0, float("nan")], [1e308, 1e308], [0.123456789, 98.7654321, 1e-9, 3.5]]
    for partials in cases:
        for max_norm in (1.0, 0.37, 1e6):
            d = torch.tensor(partials, dtype=torch.float64, device=DEV)
            coef = torch.zeros(1, dtype=torch.float32, device=DEV)
            bad = torch.zeros(1, dtype=torch.int32, device=DEV)
            zs.zs_clip_coefficient(d, len(partials), max_norm, coef, bad)
            c_ref, bad_ref = orc.clip_coef(partials, max_norm)
            assert int(bad.item()) == bad_ref
            assert coef.cpu().numpy().view(np.uint32)[0] == np.float32(c_ref).view(np.uint32)


def _pipeline(orc, N, S, seed, max_norm_frac, poison=None, steps=2):
    plan = zs.zs_flatten_plan([N * S], world=N)
    S = plan.S
    master0 = synth.fill(S * N, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02)
    o_st = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
            for r in range(N)]
    o_full = [np.zeros(S * N, np.uint16) for _ in range(N)]
    d_st = [[to_dev(x.copy()) for x in st] for st in o_st]
    d_full = [torch.zeros(S * N, dtype=torch.int16, device=DEV) for _ in range(N)]
    ws = workspace()
    parts = torch.zeros(N, dtype=torch.float64, device=DEV)
    coef = torch.zeros(1, dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    max_norm = None
    coefs = []
    for t in range(1, steps + 1):
        local = [synth.fill(S * N, seed=seed, rank=j, step=t, bf16=True) for j in range(N)]
        if poison is not None and t == steps:
            local[poison[0]][poison[1]] = 0x7FC0
        slices = [[local[j][r * S:(r + 1) * S].copy() for j in range(N)] for r in range(N)]
        o_parts = [orc.grad_sqnorm(world=N, S=S, lo=0, hi=S, grads=slices[r]) for r in range(N)]
        if max_norm is None:
            max_norm = max_norm_frac * float(np.sqrt(sum(o_parts)))
        o_coef, o_bad = orc.clip_coef(o_parts, max_norm)
        for r in range(N):
            orc.shard_step_clipped(world=N, rank=r, S=S, lo=0, hi=S, grads=slices[r],
                                   master=o_st[r][0], m=o_st[r][1], v=o_st[r][2],
                                   full_flat=o_full[r], coef=o_coef, skip=o_bad, t=t,
                                   **oracle_hp(HP))
        d_slices = [[to_dev(x) for x in sl] for sl in slices]
        for r in range(N):
            out = parts.narrow(0, r, 1)
            zs.zs_grad_sqnorm(plan, r, 0, S, d_slices[r], zs.ZS_BF16, ws, out)
        zs.zs_clip_coefficient(parts, N, max_norm, coef, bad)
        for r in range(N):
            zs.zs_shard_step_clipped(plan, r, 0, S, d_slices[r], zs.ZS_BF16, *d_st[r], d_full[r],
                                     zs.ZS_BF16, HP, t, coef=coef, skip=bad)
        torch.cuda.synchronize()
        coefs.append((float(coef.item()), int(bad.item()), float(o_coef), o_bad))
        assert int(bad.item()) == o_bad
        g_parts = parts.cpu().numpy()
        for r in range(N):
            if np.isfinite(o_parts[r]):
                assert abs(g_parts[r] - o_parts[r]) <= sum_bound(S) * o_parts[r]
    for r in range(N):
        for name, d, ref in zip(("master", "m", "v"), d_st[r], o_st[r]):
            assert_state_close(to_host(d, np.float32), ref, f"{name}[{r}]")
        assert_params_close(to_host(d_full[r], np.uint16), o_full[r], oracle.BF16)
    plan.free()
    return coefs


def test_clipped_pipeline_matches_oracle(orc):
    """N = 4 ranks, two steps that clip (max_norm = 0.3 x the first norm)."""
    coefs = _pipeline(orc, N=4, S=50_000, seed=3, max_norm_frac=0.3)
    for c_gpu, bad_gpu, c_ref, bad_ref in coefs:
        assert bad_gpu == bad_ref == 0 and c_gpu < 1
        assert abs(c_gpu - c_ref) <= 2 * np.spacing(np.float32(c_ref))


def test_nonfinite_gradient_skips_every_rank(orc):
    """A NaN in one source rank's gradient makes the global norm non-finite;
    every rank's second step then leaves its buffers untouched."""
    coefs = _pipeline(orc, N=4, S=8192, seed=5, max_norm_frac=10.0, poison=(2, 12345))
    assert coefs[0][1] == 0 and coefs[1][1] == 1


def _chunked_oracle_sqnorm(orc, world, S, grads, chunks=16):
    """The oracle's sum over [0, S) in ordered chunks on host threads (the
    oracle itself stays single-threaded per chunk)."""
    bounds = np.linspace(0, S, chunks + 1).astype(np.int64)
    out = [0.0] * chunks

    def work(k):
        out[k] = orc.grad_sqnorm(world=world, S=S, lo=int(bounds[k]), hi=int(bounds[k + 1]),
                                 grads=grads)

    th = [threading.Thread(target=work, args=(k,)) for k in range(chunks)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    return sum(out)


def test_llama_7b_full_size_norm(orc):
    """The norm pass on a full Llama-7B shard (8 x 842M bf16 slices with 1 %
    x100 outliers) against the oracle over the same regenerated slices."""
    w = LLAMA_7B
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    rank = 3
    kw = dict(seed=w.seed, sigma=w.grad_sigma, p_limit=P, outlier_frac=w.outlier_frac,
              outlier_scale=w.outlier_scale, bf16=True)
    d = []
    for j in range(N):
        t = torch.empty(S, dtype=torch.int16, device=DEV)
        synth.fill_device(t.data_ptr(), S, index0=rank * S, rank=j, step=1,
                          cuda_stream=torch.cuda.current_stream().cuda_stream, **kw)
        d.append(t)
    got = float(gpu_sqnorm(plan, rank, 0, S, d, zs.ZS_BF16).item())
    del d
    torch.cuda.empty_cache()
    host = [synth.fill(S, index0=rank * S, rank=j, step=1, **kw) for j in range(N)]
    ref = _chunked_oracle_sqnorm(orc, N, S, host)
    assert abs(got - ref) <= sum_bound(S) * ref, (got, ref)
    plan.free()


def test_norm_argument_errors():
    plan = zs.zs_flatten_plan([4096], world=4)
    g = [torch.zeros(plan.S, dtype=torch.int16, device=DEV) for _ in range(4)]
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    small = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_grad_sqnorm(plan, 0, 0, plan.S, g, zs.ZS_BF16, small, out)
    assert e.value.status == zs.ZS_ERR_RANGE
    with pytest.raises(zs.ZsError) as e:
        zs.zs_clip_coefficient(out, 0, 1.0, out, out)
    assert e.value.status == zs.ZS_ERR_RANGE
    c = torch.zeros(1, dtype=torch.float32, device=DEV)
    f = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_clip_coefficient(out, 1, -1.0, c, f)
    assert e.value.status == zs.ZS_ERR_INVAL
    plan.free()


def test_gpt2_small_norm(orc):
    """The GPT-2-small shard (S = 15,555,072, N = 8) against the oracle's sum
    over 16 chunks."""
    w = GPT2_SMALL
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    rank = 5
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    for j, g in enumerate(grads):
        synth.fill_device(g.data_ptr(), S, index0=rank * S, seed=w.seed, rank=j, step=1,
                          sigma=w.grad_sigma, p_limit=P, bf16=True, cuda_stream=stream)
    got = float(gpu_sqnorm(plan, rank, 0, S, grads, zs.ZS_BF16).item())
    host = [synth.fill(S, index0=rank * S, seed=w.seed, rank=j, step=1, sigma=w.grad_sigma,
                       p_limit=P, bf16=True) for j in range(N)]
    ref = float(_chunked_oracle_sqnorm(orc, N, S, host))
    assert abs(got - ref) <= sum_bound(S) * ref, (got, ref)
    plan.free()
