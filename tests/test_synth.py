"""The synthetic input generator: counter-based determinism, distribution,
outliers, tail pad, and its bf16 rounding against PyTorch's."""
import math

import numpy as np
import torch

import synth


def test_counter_based_slices_agree():
    full = synth.fill(100_000, seed=7, rank=3, step=2, sigma=1e-3, bf16=True)
    part = synth.fill(1000, index0=5000, seed=7, rank=3, step=2, sigma=1e-3, bf16=True,
                      p_limit=100_000, threads=1)
    assert np.array_equal(full[5000:6000], part)
    idx = np.array([0, 17, 99_999, 5000])
    at = synth.at(idx, seed=7, rank=3, step=2, sigma=1e-3, bf16=True, p_limit=100_000)
    assert np.array_equal(at, full[idx])


def test_streams_steps_ranks_differ():
    a = synth.fill(1000, seed=0, rank=0, step=1)
    for kw in (dict(rank=1, step=1), dict(rank=0, step=2), dict(rank=0, step=1, seed=1),
               dict(rank=0, step=1, stream=synth.STREAM_MASTER)):
        kw.setdefault("seed", 0)
        assert not np.array_equal(a, synth.fill(1000, **kw))


def test_lockstep_fill_equals_scalar_definition():
    """Contiguous fills run 16 elements in lockstep; gathers at arbitrary
    indices run the definition one element at a time. Both give the same bits,
    for both streams, with outliers, across the tail pad and a ragged end."""
    rng = np.random.default_rng(11)
    for trial in range(12):
        n = int(rng.integers(1, 40_000))
        index0 = int(rng.integers(0, 1 << 40))
        p_limit = index0 + int(rng.integers(0, n + 40))
        kw = dict(seed=int(rng.integers(0, 1 << 32)), rank=int(rng.integers(0, 64)),
                  step=int(rng.integers(1, 20)), p_limit=p_limit, bf16=bool(trial % 2),
                  stream=synth.STREAM_GRAD if trial % 3 else synth.STREAM_MASTER,
                  sigma=float(rng.choice([1e-3, 0.02, 1.0])))
        if trial % 4 == 0:
            kw.update(outlier_frac=0.01, outlier_scale=100.0)
        a = synth.fill(n, index0=index0, threads=3, **kw)
        b = synth.at(np.arange(index0, index0 + n), threads=2, **kw)
        assert np.array_equal(a, b), trial


def test_threads_do_not_change_values():
    a = synth.fill(50_000, seed=4, threads=1)
    b = synth.fill(50_000, seed=4, threads=7)
    assert np.array_equal(a, b)


def test_normal_moments():
    n = 2_000_000
    x = synth.fill(n, seed=0, stream=synth.STREAM_MASTER, sigma=1.0).astype(np.float64)
    se = 1 / math.sqrt(n)
    assert abs(x.mean()) < 5 * se
    assert abs(x.var() - 1) < 5 * math.sqrt(2) * se
    assert abs((x ** 3).mean()) < 5 * math.sqrt(15) * se
    assert abs((x ** 4).mean() - 3) < 5 * math.sqrt(96) * se
    # Tail mass beyond 2 sigma: 4.55%.
    assert abs((np.abs(x) > 2).mean() - 0.0455003) < 5 * math.sqrt(0.0455 / n)


def test_outlier_fraction_and_scale():
    n = 1_000_000
    plain = synth.fill(n, seed=0, rank=1, step=1, sigma=1e-3)
    out = synth.fill(n, seed=0, rank=1, step=1, sigma=1e-3, outlier_frac=0.01,
                     outlier_scale=100.0)
    sel = plain != out
    frac = sel.mean()
    assert abs(frac - 0.01) < 5 * math.sqrt(0.01 / n)
    np.testing.assert_allclose(out[sel], plain[sel] * 100, rtol=2 ** -23)


def test_tail_pad_is_zero():
    x = synth.fill(1000, seed=0, p_limit=900, bf16=True)
    assert not x[900:].any() and x[:900].all()


def test_log_series_accuracy():
    L = synth.lib()
    for v in np.geomspace(1e-30, 1 - 1e-12, 2000):
        assert abs(L.syn_log_host(float(v)) - math.log(v)) <= 4e-16 * max(1, abs(math.log(v)))


def test_bf16_matches_torch_rounding():
    x = synth.fill(200_000, seed=3, sigma=1e-3)
    b = synth.fill(200_000, seed=3, sigma=1e-3, bf16=True)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)
