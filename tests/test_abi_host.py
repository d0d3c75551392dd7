"""The C-ABI library on the host, no GPU: it loads, exports every function
include/zs.h declares, its planner agrees with the oracle's, and argument
errors come back as status codes before any CUDA call."""
import itertools
import os
import re

import numpy as np
import pytest

import fsdp_sharded_mixed_gb300 as zs
from synth.workloads import GPT2_SMALL, LLAMA_7B, QWEN25_3B, TINY

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "zs.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(zs_[a-z_0-9]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_symbols_are_exported():
    names = declared_functions()
    assert "zs_shard_step" in names and "zs_flatten_plan" in names
    assert "zs_gather_assemble" in names
    L = zs.lib()
    for name in names:
        assert hasattr(L, name), f"{name} declared in zs.h but not exported"
    assert set(names) == set(zs.EXPORTS), "binding and header disagree"


def test_status_strings():
    L = zs.lib()
    for st in range(0, -8, -1):
        assert L.zs_status_string(st).decode() not in ("", "unknown status")
    assert zs.zs_version() == "0.1.0"


def _plans_equal(orc, numels, ties, world, align, bucket):
    o = orc.plan(numels, ties, world=world, align=align, bucket_elems=bucket)
    p = zs.zs_flatten_plan(numels, ties, world=world, align_elems=align, bucket_elems=bucket)
    assert (p.P, p.P_pad, p.S) == (o["P"], o["P_pad"], o["S"])
    assert zs.zs_plan_offsets(p) == list(o["offsets"])
    assert [zs.zs_plan_bucket_range(p, b) for b in range(p.n_buckets)] == o["buckets"]
    for r in range(world):
        for b, (flo, fhi) in enumerate(o["buckets"]):
            assert zs.zs_plan_bucket(p, b, r) == orc.shard_range(flo, fhi, r, o["S"])
    p.free()


def test_planner_matches_oracle_bruteforce(orc):
    rng = np.random.default_rng(3)
    for k in range(0, 4):
        for numels in itertools.product(range(1, 4), repeat=k):
            for world in (1, 2, 3, 4):
                ties = [-1] * k
                if k >= 2 and numels[0] == numels[k - 1]:
                    ties[k - 1] = 0
                for bucket in (0, 1, 3, 5):
                    _plans_equal(orc, list(numels), ties, world, int(rng.integers(1, 5)), bucket)


@pytest.mark.parametrize("w", [TINY, GPT2_SMALL, QWEN25_3B, LLAMA_7B], ids=lambda w: w.key)
def test_planner_matches_oracle_workloads(orc, w):
    _plans_equal(orc, w.numels, w.tied_to, w.world, w.align, w.bucket_elems)


def test_plan_errors():
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([4, 5], [-1, 0])  # tie with a different numel
    assert e.value.status == zs.ZS_ERR_INVAL
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([4, 4], [-1, 1])  # tie to itself / later param
    assert e.value.status == zs.ZS_ERR_INVAL
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([4], world=0)
    assert e.value.status == zs.ZS_ERR_RANGE
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([4], world=zs.ZS_MAX_WORLD + 1)
    assert e.value.status == zs.ZS_ERR_RANGE
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([-1])
    assert e.value.status == zs.ZS_ERR_INVAL
    with pytest.raises(zs.ZsError) as e:
        zs.zs_flatten_plan([2 ** 62, 2 ** 62])
    assert e.value.status == zs.ZS_ERR_RANGE
    p = zs.zs_flatten_plan([3, 4], world=2, align_elems=8, bucket_elems=4)
    with pytest.raises(zs.ZsError):
        zs.zs_plan_bucket(p, p.n_buckets, 0)
    with pytest.raises(zs.ZsError):
        zs.zs_plan_bucket(p, 0, 2)


def test_plan_double_free_is_detected():
    p = zs.zs_flatten_plan([10], world=2)
    h = p.handle
    p.free()
    L = zs.lib()
    assert L.zs_plan_free(h) == zs.ZS_ERR_INVAL
    assert L.zs_plan_info(h, None, None, None, None, None, None) == zs.ZS_ERR_INVAL
    assert L.zs_plan_free(None) == zs.ZS_ERR_INVAL


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _step(p, **kw):
    args = dict(rank=0, lo=0, hi=p.S, grad_slices=[16 * (j + 1) * 4096 for j in range(p.world)],
                grad_dtype=zs.ZS_BF16, master=16 * 1_000_000, exp_avg=16 * 2_000_000,
                exp_avg_sq=16 * 3_000_000, full_flat=16 * 4_000_000, param_dtype=zs.ZS_BF16,
                hp=HP, step=1, stream=0)
    args.update(kw)
    zs.zs_shard_step(p, **args)


@pytest.mark.parametrize("kw,status", [
    (dict(rank=4), zs.ZS_ERR_RANGE),
    (dict(rank=-1), zs.ZS_ERR_RANGE),
    (dict(lo=5, hi=4), zs.ZS_ERR_RANGE),
    (dict(hi=10 ** 9), zs.ZS_ERR_RANGE),
    (dict(step=0), zs.ZS_ERR_RANGE),
    (dict(grad_dtype=zs.ZS_FP24), zs.ZS_ERR_INVAL),
    (dict(param_dtype=7), zs.ZS_ERR_INVAL),
    (dict(hp=dict(HP, beta1=1.0)), zs.ZS_ERR_INVAL),
    (dict(hp=dict(HP, eps=-1.0)), zs.ZS_ERR_INVAL),
    (dict(hp=dict(HP, lr=float("nan"))), zs.ZS_ERR_INVAL),
    (dict(master=16 * 1_000_000 + 4), zs.ZS_ERR_ALIGN),
    (dict(grad_slices=[None, 16, 32, 48]), zs.ZS_ERR_INVAL),
    (dict(grad_slices=[16 * 4096 + 8, 32, 48, 64]), zs.ZS_ERR_ALIGN),
    (dict(exp_avg=16 * 1_000_000 + 16), zs.ZS_ERR_INVAL),        # overlaps master
    (dict(full_flat=16 * 4096), zs.ZS_ERR_INVAL),                # overlaps slice 0
])
def test_step_argument_errors(kw, status):
    p = zs.zs_flatten_plan([1000], world=4)
    with pytest.raises(zs.ZsError) as e:
        _step(p, **kw)
    assert e.value.status == status, str(e.value)


def test_empty_range_is_a_no_op():
    p = zs.zs_flatten_plan([1000], world=4)
    _step(p, lo=7, hi=7, master=None)  # nothing to do: no pointer is touched


def test_null_plan_rejected():
    L = zs.lib()
    assert L.zs_shard_step(None, 0, 0, 1, None, 0, None, None, None, None, 0, None, 1,
                           None) == zs.ZS_ERR_INVAL
    assert L.zs_gather_assemble(None, 0, None, None, 0, None, None) == zs.ZS_ERR_INVAL


def test_selftest_and_step_path_arguments():
    """Argument checks of the wait self-test and the step-path switch, on the
    host (no kernel is launched for a rejected call)."""
    L = zs.lib()
    assert L.zs_selftest_wait_timeout(0, None) == zs.ZS_ERR_RANGE
    assert L.zs_selftest_wait_timeout((1 << 20) + 1, None) == zs.ZS_ERR_RANGE
    old = zs.zs_set_step_path(zs.STEP_PATH_DIRECT)
    assert zs.zs_set_step_path(zs.STEP_PATH_STAGED) == zs.STEP_PATH_DIRECT
    assert zs.zs_set_step_path(old) == zs.STEP_PATH_STAGED
    with pytest.raises(ValueError):
        zs.zs_set_step_path(5)
    assert L.zs_set_step_path(-1) == -1


def test_checked_library_exports_and_flags():
    """Both builds export the same symbols; only libzs_checked.so says it is
    the bounds-checked build and accepts the window self-test (host-side
    calls, no kernel)."""
    import ctypes
    names = declared_functions()
    checked = ctypes.CDLL(zs.CHECKED_LIB_PATH)
    for name in names:
        assert hasattr(checked, name), f"{name} missing from libzs_checked.so"
    checked.zs_bounds_checked.restype = ctypes.c_int32
    checked.zs_selftest_bounds_window.argtypes = [ctypes.c_int64]
    assert checked.zs_bounds_checked() == 1
    assert checked.zs_selftest_bounds_window(-1) == zs.ZS_ERR_RANGE
    assert checked.zs_selftest_bounds_window(0) == zs.ZS_OK
    L = zs.lib()
    assert zs.lib_path() == zs.LIB_PATH and not zs.zs_bounds_checked()
    assert L.zs_selftest_bounds_window(3) == zs.ZS_ERR_UNSUPPORTED


def test_strided_buffers_refused():
    """The binding passes dense buffers only: a strided view is refused before
    the library is called."""
    import numpy as np
    import torch
    plan = zs.zs_flatten_plan([1000], world=4)
    a = np.zeros((plan.S, 2), np.float32)[:, 0]
    with pytest.raises(ValueError):
        zs.zs_checkpoint_save(plan, 0, a, a, a, 1, "/nonexistent/never-written", stream=0)
    t = torch.zeros(plan.S * 2)[::2]
    with pytest.raises(ValueError):
        _step(plan, master=t)
    plan.free()


def test_short_buffers_refused():
    """A tensor or array shorter than the bytes a call touches is refused by
    the binding (raw addresses go to the library, which checks device
    allocations where the driver can tell)."""
    import numpy as np
    import torch
    plan = zs.zs_flatten_plan([1000], world=4)
    short = np.zeros(plan.S - 1, np.float32)
    with pytest.raises(ValueError, match="master holds"):
        zs.zs_checkpoint_save(plan, 0, short, short, short, 1, "/nonexistent/never-written",
                              stream=0)
    with pytest.raises(ValueError, match="grad_slices\\[2\\]"):
        _step(plan, grad_slices=[16, 32, torch.zeros(plan.S - 1, dtype=torch.int16), 48])
    with pytest.raises(ValueError, match="output"):
        _step(plan, full_flat=torch.zeros(plan.P_pad - 1, dtype=torch.int16))
    _step(plan, lo=3, hi=3, master=np.zeros(1, np.float32))   # empty range: nothing checked
    plan.free()


def test_buffers_marshalled_once():
    """zs.Buffers holds a slice list's addresses in a C array, checked once:
    accepted wherever a list of slices is, and a short one is still refused."""
    import torch
    plan = zs.zs_flatten_plan([1000], world=4)
    addrs = [16 * (j + 1) * 4096 for j in range(4)]
    b = zs.Buffers(addrs)
    assert len(b) == 4 and b.min_nbytes is None and list(b.array) == addrs
    with pytest.raises(zs.ZsError) as e:
        _step(plan, grad_slices=b, rank=4)          # reaches the library: rank out of range
    assert e.value.status == zs.ZS_ERR_RANGE
    short = zs.Buffers([torch.zeros(plan.S, dtype=torch.int16) for _ in range(3)] +
                       [torch.zeros(plan.S - 1, dtype=torch.int16)])
    assert short.min_nbytes == (plan.S - 1) * 2
    with pytest.raises(ValueError, match="gradient slice holds"):
        _step(plan, grad_slices=short)
    with pytest.raises(ValueError):
        zs.Buffers([torch.zeros(2 * plan.S, dtype=torch.int16)[::2]])
    plan.free()
