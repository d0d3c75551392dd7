"""GPU parity of per-parameter row sharding (FSDP2): copy-in (and resharding
to a smaller world), the emulated AllGather, copy-out into parameters, and the
shard step on the row layout, all against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import oracle
import synth
from gpu_util import DEV, assert_params_close, assert_state_close, oracle_hp, to_dev, to_host
from synth.workloads import LLAMA_7B

pytestmark = pytest.mark.gpu

DT = {2: zs.ZS_BF16, 4: zs.ZS_FP32, 3: zs.ZS_FP24}


def _random_params(rng, k, big=False):
    dims, numels, ties = [], [], []
    for i in range(k):
        if i > 1 and rng.random() < 0.2:
            j = int(rng.integers(0, i))
            while ties[j] >= 0:
                j = ties[j]
            dims.append(dims[j]); numels.append(numels[j]); ties.append(j)
            continue
        d = int(rng.integers(0, 3000 if big else 70))
        w = int(rng.integers(1, 40))
        dims.append(d); numels.append(d * w); ties.append(-1)
    return dims, numels, ties


@pytest.mark.parametrize("seed", range(12))
def test_rows_round_trip_and_reshard(orc, seed):
    rng = np.random.default_rng(900 + seed)
    N = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    M = int(rng.integers(1, N + 1))
    eb = int(rng.choice([2, 2, 4, 3]))
    dims, numels, ties = _random_params(rng, int(rng.integers(1, 9)), big=seed % 2 == 0)
    align = int(rng.choice([128, 16, 1]))
    plan = zs.zs_rows_plan(dims, numels, ties, world=N, align_elems=align)
    rp = orc.rows_plan(dims, numels, ties, world=N, align=align)
    assert plan.S == rp["S"] and zs.zs_plan_offsets(plan) == list(rp["offsets"])
    S = plan.S
    full = [None if t >= 0 else rng.integers(0, 256, size=n * eb, dtype=np.uint8)
            for n, t in zip(numels, ties)]
    d_full = [None if f is None else to_dev(f) for f in full]
    # Copy-in for every rank into one rank-major buffer (the emulated AllGather
    # of the locals is zs_gather_assemble of per-rank buffers).
    locals_ = [torch.full((max(S, 1) * eb,), 0xEE, dtype=torch.uint8, device=DEV)
               for _ in range(N)]
    for r in range(N):
        zs.zs_shard_rows(plan, r, d_full, DT[eb], locals_[r])
        ref = np.zeros(S * eb, np.uint8)
        orc.shard_rows(rp, r, eb, full, ref)
        assert np.array_equal(to_host(locals_[r], np.uint8)[:S * eb], ref), f"rank {r}"
    gathered = torch.full((N * S * eb + 64,), 0x77, dtype=torch.uint8, device=DEV)
    zs.zs_gather_assemble(plan, 0, [None] + locals_[1:], gathered, DT[eb])
    gathered.narrow(0, 0, S * eb).copy_(locals_[0].narrow(0, 0, S * eb))
    outs = [None if f is None else torch.full((f.size,), 0xAB, dtype=torch.uint8, device=DEV)
            for f in full]
    zs.zs_unshard(plan, gathered, DT[eb], outs)
    torch.cuda.synchronize()
    for f, o in zip(full, outs):
        if f is not None:
            assert np.array_equal(to_host(o, np.uint8), f)
    assert bool((gathered[N * S * eb:] == 0x77).all())
    # reshard_after_forward = M: the M-way chunks from the full parameters.
    planM = zs.zs_rows_plan(dims, numels, ties, world=M, align_elems=align)
    rpM = orc.rows_plan(dims, numels, ties, world=M, align=align)
    for r in range(M):
        loc = torch.zeros(max(planM.S, 1) * eb, dtype=torch.uint8, device=DEV)
        zs.zs_shard_rows(planM, r, outs, DT[eb], loc)
        ref = np.zeros(planM.S * eb, np.uint8)
        orc.shard_rows(rpM, r, eb, full, ref)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(loc, np.uint8)[:planM.S * eb], ref), f"M={M} rank {r}"
    plan.free()
    planM.free()


def test_rows_step_gather_unshard_matches_oracle(orc):
    """Two steps of the row-layout pipeline (each rank's slices are its chunks of
    the source ranks' gradients; step; gather; copy-out) against the oracle's."""
    rng = np.random.default_rng(77)
    dims, numels, ties = [1000, 96, 96, 3, 50, 4096], [64000, 6144, 6144, 192, 50, 4096 * 33], \
        [-1, -1, 1, -1, -1, -1]
    N = 4
    plan = zs.zs_rows_plan(dims, numels, ties, world=N, align_elems=128)
    rp = orc.rows_plan(dims, numels, ties, world=N, align=128)
    S = plan.S
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    master_params = [None if t >= 0 else synth.fill(n, seed=i, stream=synth.STREAM_MASTER,
                                                     sigma=0.02)
                     for i, (n, t) in enumerate(zip(numels, ties))]
    o_state, d_state = [], []
    for r in range(N):
        loc = np.zeros(S * 4, np.uint8)
        orc.shard_rows(rp, r, 4, [None if x is None else x.view(np.uint8) for x in master_params],
                       loc)
        st = [loc.view(np.float32).copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
        o_state.append(st)
        d_state.append([to_dev(x.copy()) for x in st])
    d_full = [torch.zeros(S * N, dtype=torch.int16, device=DEV) for _ in range(N)]
    o_full = [np.zeros(S * N, np.uint16) for _ in range(N)]
    for t in (1, 2):
        src = [[None if tt >= 0 else synth.fill(n, seed=100 * t + j, rank=i, bf16=True)
                for i, (n, tt) in enumerate(zip(numels, ties))] for j in range(N)]
        for r in range(N):
            slices = []
            for j in range(N):
                loc = np.zeros(S * 2, np.uint8)
                orc.shard_rows(rp, r, 2, [None if x is None else x.view(np.uint8) for x in src[j]],
                               loc)
                slices.append(loc.view(np.uint16).copy())
            zs.zs_shard_step(plan, r, 0, S, [to_dev(x) for x in slices], zs.ZS_BF16,
                             *d_state[r], d_full[r], zs.ZS_BF16, hp, t)
            orc.shard_step(world=N, rank=r, S=S, lo=0, hi=S, grads=slices, master=o_state[r][0],
                           m=o_state[r][1], v=o_state[r][2], full_flat=o_full[r], t=t,
                           **oracle_hp(hp))
        gathered = torch.zeros(S * N, dtype=torch.int16, device=DEV)
        zs.zs_gather_assemble(plan, 0, [d_full[j].narrow(0, j * S, S) for j in range(N)], gathered,
                              zs.ZS_BF16)
        gathered.narrow(0, 0, S).copy_(d_full[0].narrow(0, 0, S))
        outs = [None if tt >= 0 else torch.zeros(n, dtype=torch.int16, device=DEV)
                for n, tt in zip(numels, ties)]
        zs.zs_unshard(plan, gathered, zs.ZS_BF16, outs)
        o_gathered = np.concatenate([o_full[j][j * S:(j + 1) * S] for j in range(N)])
        o_outs = [None if tt >= 0 else np.zeros(n, np.uint16) for n, tt in zip(numels, ties)]
        orc.unshard(rp, o_gathered.view(np.uint8), 2,
                    [None if x is None else x.view(np.uint8) for x in o_outs])
        torch.cuda.synchronize()
        for d, o in zip(outs, o_outs):
            if o is not None:
                assert assert_params_close(to_host(d, np.uint16), o, oracle.BF16) == 0
        for r in range(N):
            for name, d, o in zip(("master", "m", "v"), d_state[r], o_state[r]):
                assert assert_state_close(to_host(d, np.float32), o, name) == 0
    plan.free()


def test_llama_block_unit_copy_out(orc):
    """One Llama-7B transformer block as a wrap unit (9 parameters, N = 8):
    gathered buffer -> parameters, every element against the oracle."""
    ps = LLAMA_7B.params[1:10]
    dims = [p.shape[0] for p in ps]
    numels = [p.numel for p in ps]
    N = 8
    plan = zs.zs_rows_plan(dims, numels, None, world=N, align_elems=128)
    rp = orc.rows_plan(dims, numels, None, world=N, align=128)
    S = plan.S
    g = synth.fill(N * S, seed=4, rank=0, step=1, bf16=True)
    d_g = to_dev(g)
    outs = [torch.empty(n, dtype=torch.int16, device=DEV) for n in numels]
    zs.zs_unshard(plan, d_g, zs.ZS_BF16, outs)
    refs = [np.zeros(n, np.uint16) for n in numels]
    orc.unshard(rp, g.view(np.uint8), 2, [x.view(np.uint8) for x in refs])
    torch.cuda.synchronize()
    for d, r in zip(outs, refs):
        assert np.array_equal(to_host(d, np.uint16), r)
    plan.free()


def test_rows_argument_errors():
    flat = zs.zs_flatten_plan([100], world=2)
    rows = zs.zs_rows_plan([10], [100], world=2)
    buf = torch.zeros(1024, dtype=torch.int16, device=DEV)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_unshard(flat, buf, zs.ZS_BF16, [buf])
    assert e.value.status == zs.ZS_ERR_UNSUPPORTED
    L = zs.lib()
    import ctypes
    srcs = (ctypes.c_void_p * 2)(None, None)
    views = (ctypes.c_void_p * 1)()
    assert L.zs_gather_assemble(rows.handle, 0, srcs, buf.data_ptr(), zs.ZS_BF16, views,
                                None) == zs.ZS_ERR_UNSUPPORTED
    small = torch.zeros(10, dtype=torch.int16, device=DEV)
    torch.cuda.synchronize()
    with pytest.raises(zs.ZsError):   # params_out overlaps the gathered buffer
        zs.zs_unshard(rows, buf, zs.ZS_BF16, [buf.narrow(0, 8, 100)])
    with pytest.raises(zs.ZsError):   # rank out of range
        zs.zs_shard_rows(rows, 2, [small], zs.ZS_BF16, buf)
    flat.free()
    rows.free()


def test_fsdp1_flat_units_gather(orc):
    """FSDP1's layout, a FlatParameter per wrap unit: each of two Llama-7B
    transformer blocks gets its own flat plan over N = 8 ranks; the ranks'
    shards of each unit are assembled into the unit's flat buffer by
    zs_gather_assemble (the AllGather's result) and every view lands on the
    oracle's offsets, bytes identical to the oracle's gather."""
    from synth.workloads import wrap_units
    N = 8
    for idx in wrap_units(LLAMA_7B)[:2]:
        numels = [LLAMA_7B.params[i].numel for i in idx]
        plan = zs.zs_flatten_plan(numels, world=N, align_elems=128)
        op = orc.plan(numels, None, world=N, align=128)
        S = plan.S
        assert (S, plan.P_pad) == (op["S"], op["P_pad"])
        shards = [synth.fill(S, index0=j * S, seed=21, rank=j, step=idx[0], p_limit=plan.P,
                             bf16=True) for j in range(N)]
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=DEV)
        full.narrow(0, 3 * S, S).copy_(to_dev(shards[3]))        # rank 3's own slot
        views = zs.zs_gather_assemble(plan, 3, [to_dev(x) for x in shards], full, zs.ZS_BF16)
        ref = np.zeros(plan.P_pad, np.uint16)
        orc.gather(world=N, S=S, elem_size=2, shards=shards, full_flat=ref)
        torch.cuda.synchronize()
        assert np.array_equal(to_host(full, np.uint16), ref)
        base = full.data_ptr()
        assert [(v - base) // 2 for v in views] == list(op["offsets"])
        plan.free()
