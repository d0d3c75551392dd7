"""The sharded checkpoint (zs_checkpoint_save / zs_checkpoint_load) on
host-resident state, no GPU: restores into other world sizes and layouts
against the oracle's definition of a restore, byte for byte, and fault
injection on the files (truncation, flipped bits, wrong order, mixed steps,
another parameter list, missing files)."""
import os

import numpy as np
import pytest

import fsdp_sharded_mixed_gb300 as zs
import synth
from synth.workloads import TINY


def _layout_pair(o, dims, numels, ties, kind, world, align):
    """(library plan, oracle layout) of one kind."""
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
        d = int(rng.integers(0, 300))
        dims.append(d); numels.append(d * int(rng.integers(1, 700)))
        ties.append(-1)
    return dims, numels, ties


def _state(rng, S):
    """Three fp32 arrays of arbitrary bit patterns (NaN payloads, -0, denormals):
    a restore moves bytes and must keep every one."""
    return [rng.integers(0, 2 ** 32, size=S, dtype=np.uint32).view(np.float32) for _ in range(3)]


def _save_all(plan, states, d, tag, step):
    paths = []
    for r, st in enumerate(states):
        p = os.path.join(d, f"{tag}.rank{r}")
        zs.zs_checkpoint_save(plan, r, *st, step, p)
        paths.append(p)
    return paths


@pytest.mark.parametrize("seed", range(10))
def test_restore_other_world_and_layout(orc, tmp_path, seed):
    rng = np.random.default_rng(3100 + seed)
    dims, numels, ties = _random_list(rng)
    kinds = ["flat", "rows"]
    ka, kb = kinds[seed % 2], kinds[(seed // 2) % 2]
    N, M = int(rng.choice([1, 2, 3, 4, 8])), int(rng.choice([1, 2, 3, 5, 8]))
    pa, la = _layout_pair(orc, dims, numels, ties, ka, N, int(rng.choice([1, 16, 128])))
    pb, lb = _layout_pair(orc, dims, numels, ties, kb, M, int(rng.choice([1, 16, 128])))
    states = [_state(rng, pa.S) for _ in range(N)]
    # the old shards must hold zero padding, as every real state does: take the
    # global tensors' own cut of the random values
    for k in range(3):
        cut = [orc.reshard(la, [s[k] for s in states], la, r) for r in range(N)]
        for r in range(N):
            states[r][k] = cut[r]
    paths = _save_all(pa, states, str(tmp_path), "a", 7 + seed)
    for r in range(M):
        got = [np.full(pb.S, np.nan, np.float32) for _ in range(3)]
        step = zs.zs_checkpoint_load(pb, r, paths, *got)
        assert step == 7 + seed
        for k in range(3):
            want = orc.reshard(la, [s[k] for s in states], lb, r)
            assert np.array_equal(got[k].view(np.uint32), want.view(np.uint32)), (r, k)
    info = zs.zs_checkpoint_info(paths[-1])
    assert info == dict(world=N, rank=N - 1, layout=0 if ka == "flat" else 1,
                        n_params=len(numels), P=pa.P, S=pa.S, step=7 + seed)
    pa.free()
    pb.free()


def test_next_update_equals_uninterrupted_run(orc, tmp_path):
    """Three oracle steps at N = 4, saved by the library, restored into M = 2
    by the library; the next step equals that of the run restored in memory by
    the oracle's definition (and so, by the oracle's pins, the uninterrupted
    run's update)."""
    w = TINY
    N, M = 4, 2
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
    pa = zs.zs_flatten_plan(w.numels, w.tied_to, world=N, align_elems=w.align)
    pb = zs.zs_flatten_plan(w.numels, w.tied_to, world=M, align_elems=w.align)
    la, lb = ("flat", w.numels, w.tied_to, N, w.align), ("flat", w.numels, w.tied_to, M, w.align)
    S, P = pa.S, pa.P
    st = [[synth.fill(S, index0=r * S, seed=5, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=P),
           np.zeros(S, np.float32), np.zeros(S, np.float32)] for r in range(N)]
    for t in (1, 2, 3):
        for r in range(N):
            g = [synth.fill(S, index0=r * S, seed=5, rank=j, step=t, p_limit=P, bf16=True)
                 for j in range(N)]
            orc.shard_step(world=N, rank=r, S=S, lo=0, hi=S, grads=g, master=st[r][0],
                           m=st[r][1], v=st[r][2], full_flat=np.zeros(N * S, np.uint16), t=t,
                           **hp)
    paths = _save_all(pa, st, str(tmp_path), "tiny", 3)
    for q in range(M):
        mem = [orc.reshard(la, [s[k] for s in st], lb, q) for k in range(3)]
        disk = [np.empty(pb.S, np.float32) for _ in range(3)]
        assert zs.zs_checkpoint_load(pb, q, paths, *disk) == 3
        g = [synth.fill(pb.S, index0=q * pb.S, seed=6, rank=j, step=4, p_limit=P, bf16=True)
             for j in range(M)]
        fa, fb = np.zeros(M * pb.S, np.uint16), np.zeros(M * pb.S, np.uint16)
        orc.shard_step(world=M, rank=q, S=pb.S, lo=0, hi=pb.S, grads=g, master=mem[0], m=mem[1],
                       v=mem[2], full_flat=fa, t=4, **hp)
        orc.shard_step(world=M, rank=q, S=pb.S, lo=0, hi=pb.S, grads=g, master=disk[0],
                       m=disk[1], v=disk[2], full_flat=fb, t=4, **hp)
        assert np.array_equal(fa, fb)
        for a, b in zip(mem, disk):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    pa.free()
    pb.free()


@pytest.fixture
def saved(tmp_path):
    """Four ranks of a three-parameter list (S spanning several 1 MiB blocks)
    saved at step 11."""
    numels = [1_200_000, 2_000_000, 2_800_000]
    plan = zs.zs_flatten_plan(numels, world=4, align_elems=128)
    rng = np.random.default_rng(8)
    states = [_state(rng, plan.S) for _ in range(4)]
    tail = plan.P - 3 * plan.S
    for k in range(3):
        states[3][k][tail:] = 0
    paths = _save_all(plan, states, str(tmp_path), "ck", 11)
    yield plan, states, paths, numels
    plan.free()


def _load_err(plan, rank, paths):
    out = [np.empty(plan.S, np.float32) for _ in range(3)]
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_load(plan, rank, paths, *out)
    return e.value


def _flip(path, offset, mask=0x01):
    with open(path, "r+b") as f:
        f.seek(offset)
        b = f.read(1)[0]
        f.seek(offset)
        f.write(bytes([b ^ mask]))


def test_round_trip_and_unneeded_files(saved):
    plan, states, paths, _ = saved
    out = [np.empty(plan.S, np.float32) for _ in range(3)]
    # rank 1 of the same world reads only old rank 1's file (and rank 0's header)
    assert zs.zs_checkpoint_load(plan, 1, [paths[0], paths[1], None, None], *out) == 11
    for a, b in zip(out, states[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert not any(p.endswith(".part") for p in os.listdir(os.path.dirname(paths[0])))


def test_truncated_file(saved):
    plan, _, paths, _ = saved
    os.truncate(paths[2], os.path.getsize(paths[2]) - 8)
    e = _load_err(plan, 2, paths)
    assert e.status == zs.ZS_ERR_CORRUPT and "truncated" in str(e)
    os.truncate(paths[2], 100)
    assert _load_err(plan, 2, paths).status == zs.ZS_ERR_CORRUPT


@pytest.mark.parametrize("where", ["master", "exp_avg_sq", "checksum", "header", "meta"])
def test_flipped_bit(saved, where):
    plan, _, paths, _ = saved
    info_S = plan.S
    data = 4096   # the header and metadata fit in the first page
    stride = -(-info_S * 4 // 4096) * 4096
    off = {"master": data + 3 * (1 << 20) + 5,          # block 3 of master
           "exp_avg_sq": data + 2 * stride + 17,        # block 0 of exp_avg_sq
           "checksum": data + 3 * stride + 8,           # table entry of master block 1
           "header": 40,                                 # inside P_pad
           "meta": 128 + 3}[where]
    _flip(paths[1], off, 0x40)
    e = _load_err(plan, 1, paths)
    assert e.status == zs.ZS_ERR_CORRUPT, str(e)
    if where == "master":
        assert "master block 3" in str(e)
    if where == "exp_avg_sq":
        assert "exp_avg_sq block 0" in str(e)
    # ranks that do not read the damaged file are unaffected
    if where in ("master", "exp_avg_sq", "checksum"):
        out = [np.empty(plan.S, np.float32) for _ in range(3)]
        assert zs.zs_checkpoint_load(plan, 3, paths, *out) == 11


def test_files_in_the_wrong_places(saved, tmp_path):
    plan, states, paths, numels = saved
    swapped = [paths[0], paths[2], paths[1], paths[3]]
    e = _load_err(plan, 1, swapped)
    assert e.status == zs.ZS_ERR_CORRUPT and "expected rank 1" in str(e)
    # fewer paths than the saved world
    assert _load_err(plan, 0, paths[:3]).status == zs.ZS_ERR_CORRUPT
    # a needed file left out
    e = _load_err(plan, 2, [paths[0], paths[1], None, paths[3]])
    assert e.status == zs.ZS_ERR_INVAL
    # a missing file
    e = _load_err(plan, 2, [paths[0], paths[1], str(tmp_path / "nope"), paths[3]])
    assert e.status == zs.ZS_ERR_IO
    # rank 2's file from another step
    other = str(tmp_path / "later.rank2")
    zs.zs_checkpoint_save(plan, 2, *states[2], 12, other)
    e = _load_err(plan, 2, [paths[0], paths[1], other, paths[3]])
    assert e.status == zs.ZS_ERR_CORRUPT and "step 12" in str(e)


def test_other_parameter_list(saved):
    plan, _, paths, numels = saved
    other = zs.zs_flatten_plan([1_200_000, 2_000_001, 2_799_999], world=4)
    e = _load_err(other, 0, paths)
    assert e.status == zs.ZS_ERR_INVAL and "parameter 1" in str(e)
    tied = zs.zs_flatten_plan(numels + [2_000_000], [-1, -1, -1, 1], world=4)
    assert _load_err(tied, 0, paths).status == zs.ZS_ERR_INVAL
    other.free()
    tied.free()


def test_save_errors_leave_no_file(tmp_path, saved):
    plan, states, _, _ = saved
    bad = str(tmp_path / "no_such_dir" / "x")
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_save(plan, 0, *states[0], 1, bad)
    assert e.value.status == zs.ZS_ERR_IO
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_save(plan, 4, *states[0], 1, str(tmp_path / "y"))
    assert e.value.status == zs.ZS_ERR_RANGE
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_save(plan, 0, *states[0], -1, str(tmp_path / "y"))
    assert e.value.status == zs.ZS_ERR_RANGE
    assert not os.path.exists(str(tmp_path / "y"))
    out = [np.empty(plan.S, np.float32) for _ in range(3)]
    with pytest.raises(zs.ZsError) as e:   # overlapping outputs
        zs.zs_checkpoint_load(plan, 0, [str(tmp_path / "y")] * 4, out[0], out[0], out[1])
    assert e.value.status == zs.ZS_ERR_INVAL


def test_not_a_checkpoint(tmp_path, saved):
    plan, _, paths, _ = saved
    junk = str(tmp_path / "junk")
    with open(junk, "wb") as f:
        f.write(os.urandom(4096))
    assert _load_err(plan, 0, [junk] + paths[1:]).status == zs.ZS_ERR_CORRUPT
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_info(junk)
    assert e.value.status == zs.ZS_ERR_CORRUPT


def test_empty_plan_and_padding_ranks(tmp_path):
    """An empty parameter list round-trips (S = 0, no arrays); restoring 10
    elements saved by one rank into 8 ranks of 4 gives rank 2 elements 8, 9
    and two zeros of padding, and rank 7 padding only."""
    p0 = zs.zs_flatten_plan([], world=2)
    assert p0.S == 0
    paths = [str(tmp_path / f"e{r}") for r in range(2)]
    for r in range(2):
        zs.zs_checkpoint_save(p0, r, None, None, None, 5, paths[r])
    assert zs.zs_checkpoint_load(p0, 1, paths, None, None, None) == 5
    assert zs.zs_checkpoint_info(paths[0])["P"] == 0
    p1 = zs.zs_flatten_plan([10], world=1, align_elems=1)
    src = [np.arange(10, dtype=np.float32) + 100 * k for k in range(3)]
    one = str(tmp_path / "s0")
    zs.zs_checkpoint_save(p1, 0, *src, 3, one)
    p8 = zs.zs_flatten_plan([10], world=8, align_elems=4)
    assert p8.S == 4
    for rank, want in ((2, [8, 9, 0, 0]), (7, [0, 0, 0, 0])):
        out = [np.full(p8.S, np.nan, np.float32) for _ in range(3)]
        assert zs.zs_checkpoint_load(p8, rank, [one], *out) == 3
        for k in range(3):
            exp = [x + 100 * k if i < 2 and rank == 2 else 0.0 for i, x in enumerate(want)]
            assert out[k].tolist() == exp, (rank, k)
    for p in (p0, p1, p8):
        p.free()
