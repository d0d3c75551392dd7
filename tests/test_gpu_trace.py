"""The per-call trace around real device calls: one record per call of an
accumulated, clipped step with its gather, in call order and with status 0,
and the same results with tracing on as with it off (the trace is host-side
and changes no device work)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import synth
from gpu_util import DEV

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _pipeline(plan, N, S, seed):
    """Two micro-steps accumulated, the norm and clip coefficient, the
    clipped step, the gather; returns the state and the gathered buffer."""
    stream = torch.cuda.current_stream().cuda_stream
    grads = [torch.empty(S * 2, dtype=torch.uint8, device=DEV) for _ in range(N)]
    master = torch.empty(S, dtype=torch.float32, device=DEV)
    synth.fill_device(master.data_ptr(), S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02,
                      bf16=False, cuda_stream=stream)
    m = torch.zeros(S, dtype=torch.float32, device=DEV)
    v = torch.zeros(S, dtype=torch.float32, device=DEV)
    acc = torch.empty(S, dtype=torch.float32, device=DEV)
    full = torch.zeros(N * S * 2, dtype=torch.uint8, device=DEV)
    for micro in range(2):
        for j, g in enumerate(grads):
            synth.fill_device(g.data_ptr(), S, seed=seed, rank=j, step=10 + micro, sigma=1e-3,
                              bf16=True, cuda_stream=stream)
        if micro == 0:
            zs.zs_grad_accumulate(plan, 0, 0, S, grads, zs.ZS_BF16, acc, 1)
    sq = torch.zeros(1, dtype=torch.float64, device=DEV)
    zs.zs_grad_sqnorm_noalloc(plan, 0, 0, S, grads, zs.ZS_BF16, sq)
    coef = torch.zeros(1, dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    zs.zs_clip_coefficient(sq, 1, 0.5, coef, bad)
    zs.zs_shard_step_clipped(plan, 0, 0, S, grads, zs.ZS_BF16, master, m, v, full, zs.ZS_BF16,
                             HP, 1, coef, bad)
    zs.zs_shard_step_accumulated(plan, 0, 0, S, grads, zs.ZS_BF16, acc, 2, master, m, v, full,
                                 zs.ZS_BF16, HP, 2)
    srcs = [full.narrow(0, r * S * 2, S * 2) for r in range(N)]
    out = torch.zeros(N * S * 2, dtype=torch.uint8, device=DEV)
    zs.zs_gather_assemble(plan, 0, srcs, out, zs.ZS_BF16)
    torch.cuda.synchronize()
    return [t.cpu().numpy().copy() for t in (master, m, v, out)]


def test_trace_of_a_step_pipeline(tmp_path):
    N = 4
    plan = zs.zs_flatten_plan([70_000, 3_000, 50_000], world=N, align_elems=128)
    S = plan.S
    off = _pipeline(plan, N, S, seed=5)
    path = str(tmp_path / "trace")
    zs.zs_set_trace(path)
    try:
        on = _pipeline(plan, N, S, seed=5)
    finally:
        zs.zs_set_trace(None)
    for a, b in zip(off, on):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    with open(path) as f:
        lines = f.read().splitlines()
    calls = [dict(kv.split("=", 1) for kv in ln.split()) for ln in lines]
    assert [c["call"] for c in calls] == [
        "zs_grad_accumulate", "zs_grad_sqnorm_noalloc", "zs_clip_coefficient",
        "zs_shard_step_clipped", "zs_shard_step_accumulated", "zs_gather_assemble"]
    assert [int(c["seq"]) for c in calls] == list(range(6))
    assert all(c["status"] == "0" for c in calls)
    plan_ids = {c["plan"] for c in calls if c["call"] != "zs_clip_coefficient"}
    assert len(plan_ids) == 1 and "-" not in plan_ids
    clip = calls[2]
    assert clip["plan"] == "-" and clip["world"] == "1" and clip["S"] == "-1"
    for c in calls[:2] + calls[3:5]:
        assert (c["world"], c["S"], c["lo"], c["hi"], c["grad"]) == (str(N), str(S), "0",
                                                                     str(S), "bf16")
    assert [calls[3]["step"], calls[4]["step"]] == ["1", "2"]
    assert calls[5]["param"] == "bf16" and calls[5]["grad"] == "-"
    plan.free()
