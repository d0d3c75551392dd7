"""Every-element parity at full size: the CPU oracle run over a whole shard on
all host cores, chunk by chunk, untimed, and compared bit for bit with the
state the GPU left after the same steps.

The shard-local step is element-local (element i of the update reads element
i of the N slices and of master/m/v, and writes element i of master/m/v and of
the parameter slot), so the oracle's step over a chunk [c0, c1) of the shard,
given that chunk's slices, is the whole-shard step restricted to the chunk.
Each worker regenerates its chunk's inputs with the seeded host generator
(the same counter-based values the device fill wrote: the generator's global
index is the flat index, so a chunk's values do not depend on the chunking),
runs every step of the oracle on it, and compares the final master, m, v and
parameter bytes with the GPU's. The oracle and the generator are called
through ctypes, which releases the GIL, so a thread pool uses every core.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle
import synth
from gpu_util import assert_params_close, assert_state_close, oracle_hp

CHUNK = 1 << 20


def host_threads():
    return max(1, min(os.cpu_count() or 1, 64))


def oracle_chunks(orc, *, world, rank, S, P, steps, hp, grad_kw, master_kw, pdts, lo=0,
                  hi=None, check, chunk=CHUNK, threads=None):
    """Run the oracle's shard step over [lo, hi) of rank `rank`'s shard in
    chunks, `steps` steps from master ~ synth(master_kw), m = v = 0, and call
    ``check(c0, c1, master, m, v, params)`` on each chunk's final state, where
    params maps each parameter dtype in `pdts` to the bytes the last step's
    cast wrote (the states do not depend on the parameter dtype, so the last
    step runs once per dtype from the same state). Gradient slice j at step t
    is synth(grad_kw, rank=j, step=t) at the shard's global indices. Returns
    the summed results of `check`."""
    hi = S if hi is None else hi
    base = rank * S
    hpo = oracle_hp(hp)

    def work(c0, c1):
        n = c1 - c0
        master = synth.fill(n, index0=base + c0, p_limit=P, threads=1, **master_kw)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        scratch = np.zeros(n * 4, np.uint8)
        params = {}
        for t in range(1, steps + 1):
            grads = [synth.fill(n, index0=base + c0, rank=j, step=t, p_limit=P, threads=1,
                                **grad_kw) for j in range(world)]
            if t < steps:
                orc.shard_step(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=master,
                               m=m, v=v, full_flat=scratch, param_dtype=oracle.BF16, t=t, **hpo)
                continue
            for k, pdt in enumerate(pdts):
                last = k == len(pdts) - 1
                st = (master, m, v) if last else (master.copy(), m.copy(), v.copy())
                out = np.zeros(n * oracle.ELEM_BYTES[pdt], np.uint8)
                orc.shard_step(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=st[0],
                               m=st[1], v=st[2], full_flat=out, param_dtype=pdt, t=t, **hpo)
                params[pdt] = out
        return check(c0, c1, master, m, v, params)

    return run_chunks(work, lo, hi, chunk=chunk, threads=threads)


def run_chunks(work, lo, hi, chunk=CHUNK, threads=None):
    """work(c0, c1) over [lo, hi) in chunks on a thread pool; returns the sum
    of the results (the first exception raised by a worker propagates)."""
    total = 0
    ex = cf.ThreadPoolExecutor(max_workers=threads or host_threads())
    try:
        futs = [ex.submit(work, c0, min(c0 + chunk, hi)) for c0 in range(lo, hi, chunk)]
        for f in cf.as_completed(futs):
            total += f.result()
    finally:
        ex.shutdown(wait=True, cancel_futures=True)
    return total


def bitwise_check(gpu_master, gpu_m, gpu_v, gpu_params):
    """A ``check`` for oracle_chunks against whole-shard host copies of the
    GPU's final state (numpy arrays indexed by shard element; gpu_params maps
    an oracle parameter dtype to the rank's slot bytes). Asserts the parity
    gates (fp32 state within 1e-6 relative, NaN with NaN; parameters within 1
    ulp) and returns the number of elements whose bits differ anywhere."""

    def check(c0, c1, master, m, v, params):
        diff = 0
        for name, got, ref in (("master", gpu_master, master), ("exp_avg", gpu_m, m),
                               ("exp_avg_sq", gpu_v, v)):
            g = got[c0:c1]
            if not np.array_equal(g.view(np.uint32), ref.view(np.uint32)):
                diff += assert_state_close(g, ref, f"{name}[{c0}:{c1}]")
        for pdt, ref in params.items():
            eb = oracle.ELEM_BYTES[pdt]
            g = gpu_params[pdt][c0 * eb:c1 * eb]
            if not np.array_equal(g, ref):
                diff += assert_params_close(g, ref, pdt, f"params[{c0}:{c1}]")
        return diff

    return check
