"""The bounds-checked build (libzs_checked.so, kernels compiled with
ZS_BOUNDS_CHECK=1).

Run from the ordinary build, ``test_gpu_suite_under_checked_build`` runs the
GPU parity suite again in a child process that loads the checked library: every
result must still match the oracle, and after every test the device error word
must be clear (tests/conftest.py), i.e. no kernel of any entry point computed an
access outside the window its launch declares. The other tests here run only in
that child: with the window of the step, accumulation and norm kernels narrowed
by a few elements (zs_selftest_bounds_window) the checks must fire, the
accesses outside the window must not happen (the state there is untouched),
and the rest of the range must be updated as without the narrowing. Nothing
here accesses memory out of bounds: the narrowed window lies inside buffers
that cover the whole range."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import synth
from gpu_util import DEV

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
CHECKED = os.environ.get("ZS_BOUNDS_CHECK") == "1"
checked_only = pytest.mark.skipif(not CHECKED, reason="runs in the bounds-checked child")


@pytest.mark.skipif(CHECKED, reason="already the checked build")
def test_gpu_suite_under_checked_build():
    env = dict(os.environ, ZS_BOUNDS_CHECK="1")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests"), "-m", "gpu", "-x", "-q",
           "-p", "no:cacheprovider"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((p.stdout + p.stderr).splitlines()[-25:])
    assert p.returncode == 0, tail
    assert " passed" in tail and "error" not in tail.splitlines()[-1], tail


@checked_only
def test_checked_library_is_loaded():
    assert zs.lib_path() == zs.CHECKED_LIB_PATH and zs.zs_bounds_checked()


def _state(S, seed):
    master = synth.fill(S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=S)
    return [master, np.zeros(S, np.float32), np.zeros(S, np.float32)]


def _run_step(plan, grads, state, lo, hi, path, shrink):
    S = plan.S
    d = [torch.from_numpy(x.copy()).to(DEV) for x in state]
    full = torch.full((plan.P_pad,), 0x5A5A, dtype=torch.int16, device=DEV)
    old = zs.zs_set_step_path(path)
    zs.zs_selftest_bounds_window(shrink)
    try:
        zs.zs_shard_step(plan, 0, lo, hi, grads, zs.ZS_BF16, *d, full, zs.ZS_BF16, HP, 1)
        torch.cuda.synchronize()
        status = zs.ZS_OK
        try:
            zs.zs_check_device_error()
        except zs.ZsError as e:
            status = e.status
    finally:
        zs.zs_selftest_bounds_window(0)
        zs.zs_set_step_path(old)
    out = [t.cpu().numpy() for t in d] + [full[:S].cpu().numpy().view(np.uint16)]
    return status, out


@checked_only
@pytest.mark.parametrize("path", [zs.STEP_PATH_DIRECT, zs.STEP_PATH_STAGED])
@pytest.mark.parametrize("lo_off,hi_off", [(0, 0), (13, 10)])
def test_narrowed_window_flags_and_skips_step(path, lo_off, hi_off):
    """Staged with lo = 0, hi = S: whole first and last tiles fall outside the
    window, so the producer's empty-stage path runs; with ragged ends the
    element-by-element checks fire."""
    N, S = 4, 10 * 2048
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
    assert plan.S == S
    grads = [torch.from_numpy(synth.fill(S, seed=9, rank=j, step=1, bf16=True, p_limit=S)
                              .view(np.int16)).to(DEV) for j in range(N)]
    state = _state(S, 9)
    lo, hi, k = lo_off, S - hi_off, 5
    st0, ref = _run_step(plan, grads, state, lo, hi, path, 0)
    assert st0 == zs.ZS_OK
    st1, got = _run_step(plan, grads, state, lo, hi, path, k)
    assert st1 == zs.ZS_ERR_RANGE
    init = [x.view(np.uint32) for x in state] + [np.full(S, 0x5A5A, np.uint16)]
    ref = [ref[i].view(np.uint32) if i < 3 else ref[i] for i in range(4)]
    got = [got[i].view(np.uint32) if i < 3 else got[i] for i in range(4)]
    margin = 2048 if path == zs.STEP_PATH_STAGED else 16
    for name, g, r, i0 in zip(("master", "m", "v", "param"), got, ref, init):
        outside = np.r_[0:lo + k, hi - k:S]
        assert np.array_equal(g[outside], i0[outside]), name        # never touched
        inner = slice(lo + k + margin, hi - k - margin)
        assert np.array_equal(g[inner], r[inner]), name              # updated as usual
        assert np.all((g == r) | (g == i0)), name                     # nothing else written
    plan.free()


@checked_only
def test_narrowed_window_flags_accumulate_and_norm():
    N, S, k = 8, 5000, 3
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=8)
    S = plan.S
    grads = [torch.from_numpy(synth.fill(S, seed=4, rank=j, step=1, bf16=True, p_limit=S)
                              .view(np.int16)).to(DEV) for j in range(N)]
    acc0 = torch.full((S,), 7.0, dtype=torch.float32, device=DEV)
    acc1 = acc0.clone()
    sq0 = torch.zeros(1, dtype=torch.float64, device=DEV)
    sq1 = torch.zeros(1, dtype=torch.float64, device=DEV)
    zs.zs_grad_accumulate(plan, 0, 1, S, grads, zs.ZS_BF16, acc0, 0)
    zs.zs_grad_sqnorm_noalloc(plan, 0, 1, S, grads, zs.ZS_BF16, sq0)
    zs.zs_check_device_error()
    zs.zs_selftest_bounds_window(k)
    try:
        zs.zs_grad_accumulate(plan, 0, 1, S, grads, zs.ZS_BF16, acc1, 0)
        with pytest.raises(zs.ZsError) as e:
            zs.zs_check_device_error()
        assert e.value.status == zs.ZS_ERR_RANGE
        zs.zs_grad_sqnorm_noalloc(plan, 0, 1, S, grads, zs.ZS_BF16, sq1)
        with pytest.raises(zs.ZsError) as e:
            zs.zs_check_device_error()
        assert e.value.status == zs.ZS_ERR_RANGE
    finally:
        zs.zs_selftest_bounds_window(0)
    a0, a1 = acc0.cpu().numpy(), acc1.cpu().numpy()
    assert np.all(a1[:1 + k] == 7.0) and np.all(a1[S - k:] == 7.0)
    assert np.array_equal(a1[1 + k + 16:S - k - 16], a0[1 + k + 16:S - k - 16])
    assert 0.0 < float(sq1.item()) < float(sq0.item())
    plan.free()
