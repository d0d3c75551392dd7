"""GPU side of the sharded checkpoint: device-resident state saved (blocks
hashed on the device) and restored (through pinned staging) into other world
sizes and layouts, against the oracle's definition of a restore, byte for
byte; device-saved files read into host memory and the reverse (the device and
host checksums agree); the pages' resume test on the GPT-2-small list through
the CUDA step; a corrupted file on the device path."""
import os

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_gb300 as zs
import synth
from gpu_util import DEV, to_dev, to_host
from synth.workloads import GPT2_SMALL

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _pair(o, dims, numels, ties, kind, world, align):
    if kind == "flat":
        return (zs.zs_flatten_plan(numels, ties, world=world, align_elems=align),
                ("flat", numels, ties, world, align))
    return (zs.zs_rows_plan(dims, numels, ties, world=world, align_elems=align),
            ("rows", o.rows_plan(dims, numels, ties, world=world, align=align)))


def _random_list(rng):
    dims, numels, ties = [], [], []
    for i in range(int(rng.integers(1, 8))):
        if i > 1 and rng.random() < 0.2:
            j = int(rng.integers(0, i))
            while ties[j] >= 0:
                j = ties[j]
            dims.append(dims[j]); numels.append(numels[j]); ties.append(j)
            continue
        d = int(rng.integers(0, 900))
        dims.append(d); numels.append(d * int(rng.integers(1, 900)))
        ties.append(-1)
    return dims, numels, ties


@pytest.mark.parametrize("seed", range(12))
def test_device_restore_other_world_and_layout(orc, tmp_path, seed):
    rng = np.random.default_rng(4100 + seed)
    dims, numels, ties = _random_list(rng)
    ka, kb = ("flat", "rows")[seed % 2], ("flat", "rows")[(seed // 2) % 2]
    N, M = int(rng.choice([1, 2, 4, 8])), int(rng.choice([1, 2, 3, 5, 8]))
    # align 1 gives shards whose byte length is not a multiple of 16 (the
    # checksum's zero-padded last word) and unaligned copies (checked on the host)
    pa, la = _pair(orc, dims, numels, ties, ka, N, int(rng.choice([1, 16, 128])))
    pb, lb = _pair(orc, dims, numels, ties, kb, M, int(rng.choice([1, 16, 128])))
    host = []
    for r in range(N):
        raw = [rng.integers(0, 2 ** 32, size=pa.S, dtype=np.uint32).view(np.float32)
               for _ in range(3)]
        host.append(raw)
    for k in range(3):   # zero padding, as real state has
        cut = [orc.reshard(la, [h[k] for h in host], la, r) for r in range(N)]
        for r in range(N):
            host[r][k] = cut[r]
    # even ranks save from the device, odd ranks from host memory
    paths = []
    for r in range(N):
        p = str(tmp_path / f"s.rank{r}")
        src = [to_dev(x) for x in host[r]] if r % 2 == 0 else host[r]
        zs.zs_checkpoint_save(pa, r, *src, 5, p)
        paths.append(p)
    for q in range(M):
        want = [orc.reshard(la, [h[k] for h in host], lb, q) for k in range(3)]
        dev = [torch.full((max(pb.S, 1),), float("nan"), device=DEV) for _ in range(3)]
        assert zs.zs_checkpoint_load(pb, q, paths, *dev) == 5
        hst = [np.full(pb.S, np.nan, np.float32) for _ in range(3)]
        assert zs.zs_checkpoint_load(pb, q, paths, *hst) == 5
        for k in range(3):
            got = to_host(dev[k], np.float32)[:pb.S]
            assert np.array_equal(got.view(np.uint32), want[k].view(np.uint32)), (q, k)
            assert np.array_equal(hst[k].view(np.uint32), want[k].view(np.uint32)), (q, k)
    pa.free()
    pb.free()


def _dev_state(plan, rank, seed):
    S, P = plan.S, plan.P
    m = synth.fill(S, index0=rank * S, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02,
                   p_limit=P)
    return [to_dev(m), torch.zeros(S, device=DEV), torch.zeros(S, device=DEV)]


def test_gpt2_resume_next_update_equals_uninterrupted(orc, tmp_path):
    """GPT-2-small list, N = 8: two CUDA steps, every rank saved; restored into
    M = 4; step 3 with every rank's gradient equal to one bf16 x (its mean is
    x at any power-of-two world) gives the uninterrupted N = 8 run's master,
    m, v and parameters bit for bit, and the restored state equals the
    oracle's restore of the saved state."""
    w = GPT2_SMALL
    N, M = 8, 4
    pa = zs.zs_flatten_plan(w.numels, w.tied_to, world=N, align_elems=w.align)
    pb = zs.zs_flatten_plan(w.numels, w.tied_to, world=M, align_elems=w.align)
    la = ("flat", w.numels, w.tied_to, N, w.align)
    lb = ("flat", w.numels, w.tied_to, M, w.align)
    S, P = pa.S, pa.P
    stream = torch.cuda.current_stream().cuda_stream
    state = [_dev_state(pa, r, w.seed) for r in range(N)]
    grads = [torch.empty(S, dtype=torch.int16, device=DEV) for _ in range(N)]
    full = torch.zeros(pa.P_pad, dtype=torch.int16, device=DEV)
    for t in (1, 2):
        for r in range(N):
            for j in range(N):
                synth.fill_device(grads[j].data_ptr(), S, index0=r * S, seed=w.seed, rank=j,
                                  step=t, sigma=w.grad_sigma, p_limit=P, bf16=True,
                                  cuda_stream=stream)
            zs.zs_shard_step(pa, r, 0, S, grads, zs.ZS_BF16, *state[r], full, zs.ZS_BF16, HP, t)
    paths = [str(tmp_path / f"gpt2.rank{r}") for r in range(N)]
    for r in range(N):
        zs.zs_checkpoint_save(pa, r, *state[r], 2, paths[r])
    saved = [[to_host(a, np.float32) for a in st] for st in state]
    # the uninterrupted run's step 3
    x = torch.empty(pa.P_pad, dtype=torch.int16, device=DEV)
    synth.fill_device(x.data_ptr(), pa.P_pad, seed=77, step=3, sigma=w.grad_sigma, p_limit=P,
                      bf16=True, cuda_stream=stream)
    full_a = torch.zeros(pa.P_pad, dtype=torch.int16, device=DEV)
    for r in range(N):
        xr = x.narrow(0, r * S, S)
        zs.zs_shard_step(pa, r, 0, S, [xr] * N, zs.ZS_BF16, *state[r], full_a, zs.ZS_BF16, HP, 3)
    # the restored run's step 3
    Sb = pb.S
    restored = [[torch.empty(Sb, device=DEV) for _ in range(3)] for _ in range(M)]
    for q in range(M):
        assert zs.zs_checkpoint_load(pb, q, paths, *restored[q]) == 2
        for k in range(3):
            want = orc.reshard(la, [s[k] for s in saved], lb, q)
            assert np.array_equal(to_host(restored[q][k], np.float32).view(np.uint32),
                                  want.view(np.uint32)), (q, k)
    full_b = torch.zeros(pb.P_pad, dtype=torch.int16, device=DEV)
    for q in range(M):
        xq = x.narrow(0, q * Sb, Sb)
        zs.zs_shard_step(pb, q, 0, Sb, [xq] * M, zs.ZS_BF16, *restored[q], full_b, zs.ZS_BF16,
                         HP, 3)
    torch.cuda.synchronize()
    # parameters (the flat buffers agree on every parameter's offset) and the
    # global master / m / v of the two runs, bit for bit
    assert torch.equal(full_a[:P], full_b[:P])
    for k in range(3):
        g_a = torch.cat([state[r][k] for r in range(N)])[:P]
        g_b = torch.cat([restored[q][k] for q in range(M)])[:P]
        assert torch.equal(g_a.view(torch.int32), g_b.view(torch.int32)), k
    pa.free()
    pb.free()


def test_device_corrupt_block_then_continue(orc, tmp_path):
    plan = zs.zs_flatten_plan([3_000_000], world=2, align_elems=128)
    S = plan.S
    st = [torch.randn(S, device=DEV) for _ in range(3)]
    paths = [str(tmp_path / f"c.rank{r}") for r in range(2)]
    for r in range(2):
        zs.zs_checkpoint_save(plan, r, *st, 1, paths[r])
    with open(paths[1], "r+b") as f:
        f.seek(4096 + (1 << 20) + 3)
        b = f.read(1)[0]
        f.seek(4096 + (1 << 20) + 3)
        f.write(bytes([b ^ 0x10]))
    out = [torch.empty(S, device=DEV) for _ in range(3)]
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_load(plan, 1, paths, *out)
    assert e.value.status == zs.ZS_ERR_CORRUPT and "master block 1" in str(e.value)
    # the context is fine: rank 0's file loads, and a step runs
    assert zs.zs_checkpoint_load(plan, 0, paths, *out) == 1
    torch.cuda.synchronize()
    for a, b in zip(out, st):
        assert torch.equal(a, b)
    g = [torch.zeros(S, dtype=torch.int16, device=DEV) for _ in range(2)]
    full = torch.zeros(2 * S, dtype=torch.int16, device=DEV)
    zs.zs_shard_step(plan, 0, 0, S, g, zs.ZS_BF16, *out, full, zs.ZS_BF16, HP, 2)
    torch.cuda.synchronize()
    plan.free()


@pytest.mark.parametrize("where", ["device-checked", "host-checked"])
def test_device_corrupt_in_reshard(tmp_path, where):
    """A restore from 2 ranks into 3: rank 1 of 3 takes flat elements
    [2M, 4M), i.e. old rank 0's bytes [8.0e6, ob) and old rank 1's [0, 4.0e6).
    Blocks lying whole inside a copy are checked on the device (old rank 0's
    master block 9), the edge blocks on the host (old rank 1's exp_avg block
    3); a flipped bit in either is reported with its block."""
    old = zs.zs_flatten_plan([6_000_000], world=2, align_elems=128)
    new = zs.zs_flatten_plan([6_000_000], world=3, align_elems=128)
    assert old.S == 3_000_064 and new.S == 2_000_000
    st = [torch.randn(old.S, device=DEV) for _ in range(3)]
    paths = [str(tmp_path / f"r.rank{r}") for r in range(2)]
    for r in range(2):
        zs.zs_checkpoint_save(old, r, *st, 4, paths[r])
    out = [torch.empty(new.S, device=DEV) for _ in range(3)]
    assert zs.zs_checkpoint_load(new, 1, paths, *out) == 4   # clean files load
    torch.cuda.synchronize()
    assert torch.equal(out[0][:old.S - 2_000_000], st[0][2_000_000:])
    assert torch.equal(out[1][old.S - 2_000_000:], st[1][:4_000_000 - old.S])
    stride = -(-old.S * 4 // 4096) * 4096
    if where == "device-checked":
        path, off, name = paths[0], 4096 + 9 * (1 << 20) + 100, "master block 9"
    else:
        path, off, name = paths[1], 4096 + stride + 3 * (1 << 20) + 100, "exp_avg block 3"
    with open(path, "r+b") as f:
        f.seek(off)
        b = f.read(1)[0]
        f.seek(off)
        f.write(bytes([b ^ 0x02]))
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_load(new, 1, paths, *out)
    assert e.value.status == zs.ZS_ERR_CORRUPT and name in str(e.value), str(e.value)
    old.free()
    new.free()


def test_device_argument_errors(tmp_path):
    plan = zs.zs_flatten_plan([4096], world=2)
    S = plan.S
    d = [torch.zeros(S, device=DEV) for _ in range(3)]
    h = [np.zeros(S, np.float32) for _ in range(3)]
    with pytest.raises(zs.ZsError) as e:   # mixed host and device arrays
        zs.zs_checkpoint_save(plan, 0, d[0], h[1], d[2], 1, str(tmp_path / "x"))
    assert e.value.status == zs.ZS_ERR_INVAL
    big = torch.zeros(S + 4, device=DEV)
    with pytest.raises(zs.ZsError) as e:   # misaligned device array
        zs.zs_checkpoint_save(plan, 0, big.narrow(0, 1, S), d[1], d[2], 1, str(tmp_path / "x"))
    assert e.value.status == zs.ZS_ERR_ALIGN
    # (A device array shorter than the shard is refused by the same allocation
    # check as zs_shard_step's, tested there with a write that could not leave
    # the allocation even if the check missed; a save reads the whole shard,
    # so it is not repeated here.)
    assert not os.path.exists(str(tmp_path / "x"))
    plan.free()


def test_staging_kept_and_released(tmp_path):
    """The pinned staging one call leaves for the next: repeated saves and
    restores through the kept set, a release, and a restore that allocates
    again all give the same bytes; releasing with nothing kept is a no-op.
    The state spans several 64 MiB staging units so that every slot is used."""
    zs.zs_checkpoint_release_staging()
    zs.zs_checkpoint_release_staging()
    S0 = 3 * (1 << 24) + 4096          # 3 arrays x ~201 MB: many staging items, no padding
    plan = zs.zs_flatten_plan([2 * S0], world=2, align_elems=128)
    S = plan.S
    assert S == S0
    rng = np.random.default_rng(77)
    src = [torch.from_numpy(rng.integers(0, 2 ** 32, size=S, dtype=np.uint32).view(np.int32))
           .to(DEV) for _ in range(3)]
    path = str(tmp_path / "r1")
    for rep in range(3):
        zs.zs_checkpoint_save(plan, 1, *src, 40 + rep, path)
        if rep == 1:
            zs.zs_checkpoint_release_staging()
        dst = [torch.zeros(S, dtype=torch.int32, device=DEV) for _ in range(3)]
        paths = [None, path]
        # rank 1 of the same world reads only old rank 1's file; paths[0] must
        # still name a file of the old world: save rank 0 as well
        zs.zs_checkpoint_save(plan, 0, *src, 40 + rep, str(tmp_path / "r0"))
        paths[0] = str(tmp_path / "r0")
        assert zs.zs_checkpoint_load(plan, 1, paths, *dst) == 40 + rep
        for a, b in zip(src, dst):
            assert torch.equal(a, b)
        del dst
    zs.zs_checkpoint_release_staging()
    plan.free()
