"""The library called from several host threads at once, each thread on its
own stream and buffers, from the first call of a fresh process (when the
per-device launch caches and the staged kernel's shared-memory opt-in are
first set): every thread's result equals the result of the same calls made
from one thread, bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading
import numpy as np
import torch
sys.path.insert(0, ROOT)
import fsdp_sharded_mixed_gb300 as zs
import synth

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
DEV = torch.device("cuda:0")
torch.zeros(1, device=DEV)

def job(k, out):
    # thread k: its own stream, plan and buffers; the step (staged or
    # register-streaming by size), a clipped accumulated step, the gather
    stream = torch.cuda.Stream()
    N = (4, 8, 16, 2)[k % 4]
    S0 = (40_000, 70_000, 150_000, 33_333)[k % 4]
    plan = zs.zs_flatten_plan([N * S0], world=N, align_elems=128)
    S = plan.S
    with torch.cuda.stream(stream):
        g = [torch.from_numpy(synth.fill(S, seed=k % 4, rank=j, step=1, bf16=True)
                              .view(np.int16)).to(DEV) for j in range(N)]
        st = [torch.from_numpy(synth.fill(S, seed=k % 4, stream=synth.STREAM_MASTER,
                                          sigma=0.02)).to(DEV),
              torch.zeros(S, device=DEV), torch.zeros(S, device=DEV)]
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        acc = torch.zeros(S, device=DEV)
        ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=DEV)
        sq = torch.zeros(1, dtype=torch.float64, device=DEV)
        coef = torch.zeros(1, dtype=torch.float32, device=DEV)
        bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    sp = stream.cuda_stream
    for t in (1, 2, 3):
        zs.zs_shard_step(plan, 0, 0, S, g, zs.ZS_BF16, *st, full, zs.ZS_BF16, HP, t, stream=sp)
    zs.zs_grad_accumulate(plan, 0, 0, S, g, zs.ZS_BF16, acc, 1, stream=sp)
    zs.zs_grad_sqnorm_accumulated(plan, 0, 0, S, g, zs.ZS_BF16, acc, 2, ws, sq, stream=sp)
    zs.zs_clip_coefficient(sq, 1, 0.5, coef, bad, stream=sp)
    zs.zs_shard_step_accumulated_clipped(plan, 0, 0, S, g, zs.ZS_BF16, acc, 2, *st, full,
                                         zs.ZS_BF16, HP, 4, coef=coef, skip=bad, stream=sp)
    srcs = [full.narrow(0, r * S, S) for r in range(N)]
    out_full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
    zs.zs_gather_assemble(plan, 0, srcs, out_full, zs.ZS_BF16, stream=sp)
    zs.zs_check_device_error(stream=sp)
    out[k] = [x.cpu().numpy().tobytes() for x in st + [out_full, sq]]

threads = 8
par, seq = {}, {}
ts = [threading.Thread(target=job, args=(k, par)) for k in range(threads)]
for t in ts:
    t.start()
for t in ts:
    t.join()
for k in range(threads):
    job(k, seq)
assert sorted(par) == list(range(threads)), sorted(par)
for k in range(threads):
    assert par[k] == seq[k], k
    assert par[k] == par[k % 4], k
print("threads ok")
'''


def test_concurrent_first_calls_match_sequential():
    code = "ROOT = %r\n" % ROOT + CHILD
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0 and "threads ok" in p.stdout, (p.stdout + p.stderr)[-3000:]
