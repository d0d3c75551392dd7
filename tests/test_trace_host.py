"""The per-call trace without a GPU: the record of each call at a collective
site, the ZS_TRACE variable with its %r / %p expansion, and finding the first
record where two gloo ranks' traces part ("从 Data Parallel 到 ZeRO/FSDP",
"训练 Hang 应按 Collective 顺序排查": log every collective in order and look
for the first place the ranks differ) — a module run twice on one rank, a
rank that stops early, and ranks that differ only in what they may differ in
(rank, range, status)."""
import os
import re
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import fsdp_sharded_mixed_gb300 as zs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
LINE = re.compile(r"seq=(\d+) call=(\w+) plan=([0-9a-f]{16}|-) world=(-?\d+) S=(-?\d+) "
                  r"rank=(-?\d+) lo=(-?\d+) hi=(-?\d+) grad=(\w+|-) param=(\w+|-) "
                  r"step=(-?\d+) status=(-?\d+)$")


def _records(path):
    with open(path) as f:
        lines = f.read().splitlines()
    out = []
    for ln in lines:
        m = LINE.match(ln)
        assert m, ln
        out.append(m.groups())
    return out


@pytest.fixture
def tracing(tmp_path):
    path = str(tmp_path / "trace.log")
    zs.zs_set_trace(path)
    try:
        yield path
    finally:
        zs.zs_set_trace(None)


def _no_op_step(plan, rank, step, at=3, **kw):
    """A step over an empty range [at, at): traced, touches no pointer."""
    args = dict(grad_slices=[16 * (j + 1) * 4096 for j in range(plan.world)],
                grad_dtype=zs.ZS_BF16, master=None, exp_avg=16 * 2_000_000,
                exp_avg_sq=16 * 3_000_000, full_flat=16 * 4_000_000, param_dtype=zs.ZS_BF16,
                hp=HP, step=step, stream=0)
    args.update(kw)
    zs.zs_shard_step(plan, rank, at, at, **args)


def test_records_of_calls(tracing, tmp_path):
    plan = zs.zs_flatten_plan([1000, 24, 777], world=4, align_elems=8)
    same = zs.zs_flatten_plan([1000, 24, 777], world=4, align_elems=8)
    other = zs.zs_flatten_plan([1000, 24, 777], world=2, align_elems=8)
    st = [np.arange(plan.S, dtype=np.float32) * (k + 1) for k in range(3)]
    ck = str(tmp_path / "ck.rank1")
    zs.zs_checkpoint_save(plan, 1, *st, 41, ck)
    back = [np.zeros(plan.S, np.float32) for _ in range(3)]
    paths = [str(tmp_path / f"ck.rank{r}") for r in range(4)]
    for r in (0, 2, 3):
        zs.zs_checkpoint_save(plan, r, *st, 41, paths[r])
    assert zs.zs_checkpoint_load(same, 1, paths, *back) == 41
    _no_op_step(plan, 2, 5)
    with pytest.raises(zs.ZsError) as e:
        _no_op_step(other, 9, 6)                         # rank out of range: still traced
    zs.zs_set_trace(None)
    _no_op_step(plan, 0, 7)                              # tracing is off: no record
    rec = _records(tracing)
    assert [int(r[0]) for r in rec] == list(range(len(rec))) and len(rec) == 7
    assert [r[1] for r in rec] == ["zs_checkpoint_save"] * 4 + ["zs_checkpoint_load",
                                                                "zs_shard_step", "zs_shard_step"]
    ids = {r[2] for r in rec[:6]}
    assert len(ids) == 1 and rec[6][2] not in ids        # same list+layout = same id
    for r in rec[:6]:
        assert (int(r[3]), int(r[4])) == (4, plan.S)
    assert (int(rec[6][3]), int(rec[6][4])) == (2, other.S)
    assert [int(r[5]) for r in rec] == [1, 0, 2, 3, 1, 2, 9]
    assert [int(r[10]) for r in rec[:5]] == [41] * 5     # the saved / restored step
    assert rec[5][6:10] == ("3", "3", "bf16", "bf16") and rec[5][10] == "5"
    assert [int(r[11]) for r in rec] == [0] * 6 + [e.value.status]


def test_env_variable_and_expansion(tmp_path):
    """ZS_TRACE is read at the first traced call; %r is RANK and %p the pid."""
    code = (
        "import fsdp_sharded_mixed_gb300 as zs, os\n"
        "p = zs.zs_flatten_plan([100], world=2)\n"
        "try:\n"
        "    zs.zs_shard_step(p, 5, 0, 1, [16, 32], zs.ZS_BF16, 64, 128, 256, 512,\n"
        "                     zs.ZS_BF16, dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,\n"
        "                     weight_decay=0.0), 1, stream=0)\n"
        "except zs.ZsError:\n"
        "    pass\n"
        "print(os.getpid())\n")
    env = dict(os.environ, ZS_TRACE=str(tmp_path / "t.%r.%p"), RANK="3",
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    pid = subprocess.run([sys.executable, "-c", code], env=env, check=True, capture_output=True,
                         text=True, timeout=300).stdout.split()[-1]
    rec = _records(str(tmp_path / f"t.3.{pid}"))
    assert len(rec) == 1 and rec[0][1] == "zs_shard_step" and rec[0][5] == "5"
    assert int(rec[0][11]) == zs.ZS_ERR_RANGE


def test_bad_trace_path_and_arguments(tmp_path):
    with pytest.raises(zs.ZsError) as e:
        zs.zs_set_trace(str(tmp_path / "no" / "such" / "dir" / "t"))
    assert e.value.status == zs.ZS_ERR_IO
    with pytest.raises(zs.ZsError) as e:
        zs.zs_trace_first_divergence([str(tmp_path / "missing.a"), str(tmp_path / "missing.b")])
    assert e.value.status == zs.ZS_ERR_IO
    L = zs.lib()
    assert L.zs_trace_first_divergence(None, 2, None, None, 0) == zs.ZS_ERR_INVAL


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_program(rank, world, port, d, scenario):
    """One rank of a data-parallel job: per step t, the step after the
    ReduceScatter (an empty range, at a rank-dependent offset) and an
    AllReduce over gloo; at the end a checkpoint. The scenario plants one
    difference between the ranks."""
    from datetime import timedelta

    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=20))
    try:
        zs.zs_set_trace(os.path.join(d, "trace.%r"))
        plan = zs.zs_flatten_plan([640, 3, 96], world=world, align_elems=8)
        for t in range(1, 5):
            if scenario == "stops" and rank == 1 and t == 4:
                zs.zs_set_trace(None)
                return                                    # this rank leaves before step 4
            fp32 = scenario == "dtype" and rank == 0 and t == 2
            _no_op_step(plan, rank, t, at=rank, grad_dtype=zs.ZS_FP32 if fp32 else zs.ZS_BF16)
            if scenario == "twice" and rank == 1 and t == 3:
                _no_op_step(plan, rank, t, at=rank)       # a module run a second time
            try:
                dist.all_reduce(torch.ones(1))            # the job's real collective
            except RuntimeError:
                assert scenario == "stops" and rank == 0  # its peer has gone
                zs.zs_set_trace(None)
                return
        st = [np.full(plan.S, rank, np.float32) for _ in range(3)]
        zs.zs_checkpoint_save(plan, rank, *st, 4, os.path.join(d, f"ck.{rank}"))
        zs.zs_set_trace(None)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run_job(tmp_path, scenario):
    ctx = mp.get_context("spawn")
    port = _free_port()
    d = str(tmp_path)
    procs = [ctx.Process(target=_rank_program, args=(r, 2, port, d, scenario)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    return [os.path.join(d, f"trace.{r}") for r in range(2)]


@pytest.mark.parametrize("scenario,seq", [("same", None), ("twice", 3), ("dtype", 1),
                                          ("stops", 3)])
def test_first_divergence_two_gloo_ranks(tmp_path, scenario, seq):
    paths = _run_job(tmp_path, scenario)
    recs = [_records(p) for p in paths]
    assert [r[5] for r in recs[1]] == ["1"] * len(recs[1])
    found = zs.zs_trace_first_divergence(paths)
    if seq is None:
        assert found is None and len(recs[0]) == len(recs[1]) == 5
        assert [r[1] for r in recs[0]] == ["zs_shard_step"] * 4 + ["zs_checkpoint_save"]
        return
    at, detail = found
    assert at == seq
    assert detail.startswith(f"record {seq}:") and paths[0] in detail and paths[1] in detail
    if scenario == "stops":
        assert len(recs[1]) == 3 and len(recs[0]) == 4 and "ends after 3 records" in detail
        assert f"seq={seq} call=zs_shard_step" in detail and "step=4" in detail
    elif scenario == "twice":
        assert "step=4" in detail and detail.count("step=3") == 1
    else:
        assert "grad=fp32" in detail and "grad=bf16" in detail
    # The detail is cut to fit a short buffer, NUL-terminated.
    L = zs.lib()
    import ctypes
    arr = (ctypes.c_char_p * 2)(*[os.fsencode(p) for p in paths])
    s = ctypes.c_int64()
    buf = ctypes.create_string_buffer(b"x" * 16, 16)
    assert L.zs_trace_first_divergence(arr, 2, ctypes.byref(s), buf, 12) == 0
    assert s.value == seq and buf.raw[11] == 0 and buf.raw[12:15] == b"xxx"
