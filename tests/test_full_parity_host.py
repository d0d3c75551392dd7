"""The chunked oracle run of the full-size GPU parity tests (full_parity.py)
is the whole-shard oracle: the step is element-local, so running it over
chunks of the shard, with each chunk's inputs regenerated at their global
indices, must give the whole-shard run's bits, for any chunk size (ragged
ones included), every parameter dtype and a rank whose shard holds the pad."""
import numpy as np
import pytest

import oracle
import synth
from full_parity import bitwise_check, oracle_chunks

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.mark.parametrize("chunk", [1 << 20, 77_777, 4096])
def test_chunked_oracle_equals_whole_shard(orc, chunk):
    N, S, rank, steps = 4, 300_000, 3, 3
    P = N * S - 1234                        # the last shard ends in the pad
    grad_kw = dict(seed=5, sigma=1e-3, bf16=True, outlier_frac=0.01, outlier_scale=100.0)
    master_kw = dict(seed=5, stream=synth.STREAM_MASTER, sigma=0.02)
    master = synth.fill(S, index0=rank * S, p_limit=P, **master_kw)
    m, v = np.zeros(S, np.float32), np.zeros(S, np.float32)
    pdts = [oracle.BF16, oracle.FP24, oracle.FP32]
    params = {}
    for t in range(1, steps + 1):
        grads = [synth.fill(S, index0=rank * S, rank=j, step=t, p_limit=P, **grad_kw)
                 for j in range(N)]
        for k, pdt in enumerate(pdts):
            last = k == len(pdts) - 1
            st = (master, m, v) if last else (master.copy(), m.copy(), v.copy())
            out = np.zeros(S * oracle.ELEM_BYTES[pdt], np.uint8)
            orc.shard_step(world=N, rank=0, S=S, lo=0, hi=S, grads=grads, master=st[0], m=st[1],
                           v=st[2], full_flat=out, param_dtype=pdt, t=t,
                           lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"], eps=HP["eps"],
                           wd=HP["weight_decay"])
            params[pdt] = out
    check = bitwise_check(master, m, v, params)
    diff = oracle_chunks(orc, world=N, rank=rank, S=S, P=P, steps=steps, hp=HP, grad_kw=grad_kw,
                         master_kw=master_kw, pdts=pdts, check=check, chunk=chunk, threads=4)
    assert diff == 0
    pad0 = P - rank * S
    assert not master[pad0:].any() and not params[oracle.BF16][2 * pad0:].any()


def test_chunked_oracle_sees_a_planted_difference(orc):
    """The comparison is not vacuous: one flipped bit in the reference state
    is reported as a differing element (within the gate, so counted)."""
    N, S, steps = 2, 50_000, 1
    grad_kw = dict(seed=6, sigma=1e-3, bf16=True)
    master_kw = dict(seed=6, stream=synth.STREAM_MASTER, sigma=0.02)
    master = synth.fill(S, p_limit=N * S, **master_kw)
    m, v = np.zeros(S, np.float32), np.zeros(S, np.float32)
    out = np.zeros(2 * S, np.uint8)
    grads = [synth.fill(S, rank=j, step=1, p_limit=N * S, **grad_kw) for j in range(N)]
    orc.shard_step(world=N, rank=0, S=S, lo=0, hi=S, grads=grads, master=master, m=m, v=v,
                   full_flat=out, t=1, lr=HP["lr"], beta1=HP["beta1"], beta2=HP["beta2"],
                   eps=HP["eps"], wd=HP["weight_decay"])
    m.view(np.uint32)[12_345] ^= 1
    check = bitwise_check(master, m, v, {oracle.BF16: out})
    diff = oracle_chunks(orc, world=N, rank=0, S=S, P=N * S, steps=steps, hp=HP,
                         grad_kw=grad_kw, master_kw=master_kw, pdts=[oracle.BF16], check=check,
                         chunk=8192, threads=2)
    assert diff == 1
