"""GPU parity at sweep points (shard size x N x incoming-gradient dtype x
parameter dtype), full size, in the launch configuration the bench's sweep
times: one tensor of N*S elements, rank 0's step, three steps; sampled
elements (and both ends of the shard) recomputed by the oracle from the
regenerated inputs, master/m/v bit for bit and the stored parameter bytes
exactly."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import DEV, assert_params_close, assert_state_close, oracle_hp

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
PDT = {2: (zs.ZS_BF16, oracle.BF16), 3: (zs.ZS_FP24, oracle.FP24), 4: (zs.ZS_FP32, oracle.FP32)}


# (S, N, slice bytes, parameter bytes, the kernel the per-call choice takes:
# (1, vector group) register-streaming, (2, tile elements) staged, None = any)
@pytest.mark.parametrize("S,N,gb,pb,kernel", [
    (1 << 26, 16, 4, 3, None),       # fp32 slices, 3-byte parameters
    (1 << 24, 64, 2, 4, (1, 16)),    # the widest world (no two staged tiles fit)
    (1 << 28, 2, 2, 3, (2, 2048)),   # N <= 2 with 3-byte parameters: staged
    (1 << 22, 8, 4, 2, None),
    (1 << 24, 16, 4, 3, (2, 1024)),  # fp32 slices on 1024-element tiles
    (1 << 24, 32, 2, 2, (2, 1024)),  # bf16 slices, N in 24..48, under 2^25: 1024-element tiles
    (1 << 26, 32, 2, 2, (1, 16)),    # the same above 2^25: register-streaming
    (1 << 28, 8, 2, 2, (2, 2048)),   # bf16, N = 8, large: staged
    (1 << 26, 4, 4, 2, (1, 16)),     # fp32 slices, N <= 4, from 2^25: register-streaming
    (1 << 24, 8, 2, 4, (2, 2048)),   # fp32 parameters under 2^26: staged
    (1 << 26, 8, 2, 4, (1, 16)),     # fp32 parameters from bf16 slices, N = 4..8, from 2^26
    (1 << 10, 4, 2, 2, None),        # the smallest point
])
def test_sweep_point_sampled(orc, S, N, gb, pb, kernel):
    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
    assert plan.S == S
    stream = torch.cuda.current_stream().cuda_stream
    bf16 = gb == 2
    grads = [torch.empty(S * gb, dtype=torch.uint8, device=DEV) for _ in range(N)]
    master = torch.empty(S, dtype=torch.float32, device=DEV)
    synth.fill_device(master.data_ptr(), S, seed=1, stream=synth.STREAM_MASTER, sigma=0.02,
                      bf16=False, cuda_stream=stream)
    m = torch.zeros(S, dtype=torch.float32, device=DEV)
    v = torch.zeros(S, dtype=torch.float32, device=DEV)
    full = torch.zeros(N * S * pb, dtype=torch.uint8, device=DEV)
    rng = np.random.default_rng(S + N)
    idx = np.unique(np.concatenate([rng.integers(0, S, size=min(S, 40_000)),
                                    np.arange(0, 32), np.arange(S - 32, S)])).astype(np.int64)
    K = idx.size
    o_master = synth.at(idx, seed=1, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=S)
    o_m, o_v = np.zeros(K, np.float32), np.zeros(K, np.float32)
    o_full = np.zeros(K * N * pb, np.uint8)
    for t in (1, 2, 3):
        for j, g in enumerate(grads):
            synth.fill_device(g.data_ptr(), S, seed=1, rank=j, step=t, sigma=1e-3, bf16=bf16,
                              cuda_stream=stream)
        zs.zs_shard_step(plan, 0, 0, S, grads, zs.ZS_BF16 if bf16 else zs.ZS_FP32, master, m, v,
                         full, PDT[pb][0], HP, t)
        if kernel is not None:
            assert zs.zs_last_step_kernel() == kernel
        g_host = [synth.at(idx, seed=1, rank=j, step=t, sigma=1e-3, bf16=bf16, p_limit=S)
                  for j in range(N)]
        orc.shard_step(world=N, rank=0, S=K, lo=0, hi=K, grads=g_host, master=o_master, m=o_m,
                       v=o_v, full_flat=o_full, param_dtype=PDT[pb][1], t=t, **oracle_hp(HP))
    torch.cuda.synchronize()
    ti = torch.from_numpy(idx).to(DEV)
    for name, d, ref in (("master", master, o_master), ("m", m, o_m), ("v", v, o_v)):
        assert assert_state_close(d[ti].cpu().numpy(), ref, name) == 0
        assert np.array_equal(d[ti].cpu().numpy().view(np.uint32), ref.view(np.uint32)), name
    # the parameter bytes of the sampled elements in rank 0's slot
    bi = (idx[:, None] * pb + np.arange(pb)[None, :]).reshape(-1)
    got = full[torch.from_numpy(bi).to(DEV)].cpu().numpy()
    want = o_full[:K * pb]
    assert assert_params_close(got, want, PDT[pb][1]) == 0
    assert np.array_equal(got, want)
    # the other ranks' slots are untouched
    assert int(full[S * pb:].count_nonzero()) == 0
    del grads, master, m, v, full
    torch.cuda.empty_cache()
    plan.free()
