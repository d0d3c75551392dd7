"""Pins: checks that tie the CPU oracle to what the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with a closed form, an invariant, a brute-force
enumeration, a value the pages print, or an exact-arithmetic reference. They
are written so that a plausible mistake in the oracle (a dropped term, a wrong
sign or index, a transposed operand) fails at least one of them; the mutation
test runs them against deliberately broken oracle builds to show it.
"""
from __future__ import annotations

import itertools
import os
from fractions import Fraction

import numpy as np

import oracle as orc
import synth
from synth.workloads import GPT2_SMALL, LLAMA_7B, QWEN25_3B, TINY, gpt2_params

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)
EPS32 = 2.0 ** -24  # unit roundoff of binary32, round to nearest
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers ----
def f32(x):
    return np.float32(x)


def to_bf16_exact(values):
    """bf16 bit patterns of values that bf16 represents exactly."""
    a = np.asarray(values, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not representable in bf16"
    return (bits >> 16).astype(np.uint16)


def bf16_to_f32(h):
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32)


def one_rank_step(o, grads, master, m, v, t, hp=HP, param_dtype=orc.BF16):
    """Run rank 0's shard step over the whole shard; return the param slot bytes."""
    S = master.size
    world = len(grads)
    eb = orc.ELEM_BYTES[param_dtype]
    full = np.zeros(world * S * eb + 16, dtype=np.uint8)
    o.shard_step(world=world, rank=0, S=S, lo=0, hi=S, grads=grads, master=master, m=m,
                 v=v, full_flat=full, param_dtype=param_dtype, t=t, **hp)
    return full[: S * eb].copy()


def nearest_even_keep_high(x, drop):
    """Exact-rational reference: the pattern with the low `drop` bits of the
    fp32 encoding cleared that is nearest to x (ties: even kept LSB), as the
    kept high bits; overflow past the largest finite gives infinity."""
    x = np.float32(x)
    if np.isnan(x):
        return None
    bits = int(np.array(x).view(np.uint32))
    sign = bits & 0x80000000
    mag_bits = bits & 0x7FFFFFFF
    if mag_bits == 0x7F800000:
        return (sign | mag_bits) >> drop
    value = Fraction(float(np.array(mag_bits, dtype=np.uint32).view(np.float32)))
    lo_bits = mag_bits & ~((1 << drop) - 1)

    def val(b):
        if b >= 0x7F800000:
            return None
        return Fraction(float(np.array(b, dtype=np.uint32).view(np.float32)))

    hi_bits = lo_bits + (1 << drop)
    lo_v = val(lo_bits)
    if lo_v == value:
        return (sign | lo_bits) >> drop
    hi_v = val(hi_bits)
    if hi_v is None:
        # Above the largest finite narrow value: nearest-even rounds to infinity
        # from the midpoint to the next (virtual) binade step on.
        ulp = Fraction(2) ** (((lo_bits >> 23) & 0xFF) - 127 - 23 + drop)
        mid = lo_v + ulp / 2
        keep_inf = value > mid or (value == mid and ((lo_bits >> drop) & 1))
        return (sign | (0x7F800000 if keep_inf else lo_bits)) >> drop
    d_lo, d_hi = value - lo_v, hi_v - value
    if d_lo < d_hi or (d_lo == d_hi and ((lo_bits >> drop) & 1) == 0):
        return (sign | lo_bits) >> drop
    return (sign | hi_bits) >> drop


def special_float_patterns():
    pats = [0x00000000, 0x80000000, 0x00000001, 0x00008000, 0x00008001, 0x00018000,
            0x007FFFFF, 0x00800000, 0x3F800000, 0x3F808000, 0x3F818000, 0x3F807FFF,
            0x3F808001, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7FFFFF, 0x7F800000,
            0xFF800000, 0x3F800080, 0x3F800180, 0x3F80007F, 0x7F7FFF80, 0x7F7FFF7F,
            0x00000080, 0x00000180, 0x807FFFFF, 0x7FC00000, 0xFFC00001, 0x7F800001,
            0xFFFFFFFF]
    return pats


# ------------------------------------------------------------- O4 AdamW ------
def pin_sign_law(o):
    """Step 1 with eps -> 0: mh = g and vh = g^2 up to rounding, so the update
    is lr*sign(g) plus the decoupled decay term p0*(1 - lr*wd)."""
    n, world = 4096, 4
    rng = np.random.default_rng(11)
    grads = [synth.fill(n, seed=5, stream=synth.STREAM_GRAD, rank=j, step=1, bf16=True)
             for j in range(world)]
    master = synth.fill(n, seed=5, stream=synth.STREAM_MASTER, sigma=0.02)
    gbar = sum(bf16_to_f32(g).astype(np.float64) for g in grads) / world
    for eps in (0.0, 1e-30):
        p = master.copy()
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        hp = dict(HP, eps=eps)
        one_rank_step(o, grads, p, m, v, 1, hp)
        live = gbar != 0
        assert live.sum() > n * 0.9
        expect = master.astype(np.float64) * (1 - HP["lr"] * HP["wd"]) - HP["lr"] * np.sign(gbar)
        err = np.abs(p.astype(np.float64) - expect)
        tol = 8 * EPS32 * (np.abs(master.astype(np.float64)) + HP["lr"])
        assert np.all(err[live] <= tol[live]), f"sign law violated (eps={eps})"
        if eps == 1e-30:
            dead = ~live
            expect_dead = (master * f32(1 - HP["lr"] * HP["wd"]))
            assert np.array_equal(p[dead], expect_dead[dead])
    _ = rng


def pin_zero_grad(o):
    """g == 0 with eps > 0: m and v stay exactly 0, the Adam term is 0 and the
    master is only decayed: p_t = p_{t-1} * fp32(1 - lr*wd), exactly."""
    n, world = 1000, 2
    master = synth.fill(n, seed=3, stream=synth.STREAM_MASTER, sigma=0.02)
    p, m, v = master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    zero = [np.zeros(n, np.uint16)] * world
    expect = master.copy()
    decay = f32(1.0 - HP["lr"] * HP["wd"])
    for t in range(1, 6):
        out = one_rank_step(o, zero, p, m, v, t)
        expect = (expect * decay).astype(np.float32)
        assert np.array_equal(m, np.zeros(n, np.float32)) and np.array_equal(v, m)
        assert np.array_equal(p, expect), "zero-gradient decay is not exact"
        assert np.array_equal(out.view(np.uint16), o.bf16(expect))
    # Pad elements (master 0, grads 0) stay exactly 0.
    p0 = np.zeros(8, np.float32)
    m0, v0 = np.zeros(8, np.float32), np.zeros(8, np.float32)
    out = one_rank_step(o, [np.zeros(8, np.uint16)] * 3, p0, m0, v0, 1)
    assert not p0.any() and not m0.any() and not v0.any() and not out.any()


def pin_constant_grad(o):
    """g == c every step, wd = 0: the moment recurrences have the closed forms
    m_t = (1-b1) c (1-b1^t)/(1-b1) and v_t = (1-b2) c^2 (1-b2^t)/(1-b2) in the
    fp32 coefficients (textbook: c(1-beta1^t), c^2(1-beta2^t)), hence m_hat = c,
    v_hat = c^2 and p_t = p_0 - lr * sum_t c/(|c|+eps), up to rounding."""
    world = 2
    cs = np.array([1.0, -1.0, 0.25, -3.0, 2.0 ** -9, -(2.0 ** -12), 0.0078125 * 3], np.float32)
    n = cs.size
    grads = [to_bf16_exact(cs)] * world
    hp = dict(HP, wd=0.0)
    p0 = np.linspace(-0.5, 0.5, n).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    c = cs.astype(np.float64)
    p_cf = p0.astype(np.float64)
    for t in range(1, 21):
        one_rank_step(o, grads, p, m, v, t, hp)
        sc = [float(x) for x in o.scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], 0.0,
                                            t, world)]
        b1, b2, omb1, omb2, bc1, bc2, lr, eps = sc[:8]
        m_cf = c * omb1 * (1 - b1 ** t) / (1 - b1)
        v_cf = c * c * omb2 * (1 - b2 ** t) / (1 - b2)
        assert np.all(np.abs(m - m_cf) <= 4 * t * EPS32 * np.abs(m_cf)), f"m off at t={t}"
        assert np.all(np.abs(v - v_cf) <= 6 * t * EPS32 * np.abs(v_cf)), f"v off at t={t}"
        # The textbook forms with the real betas (fp32 coefficient error:
        # 1-fp32(0.999) differs from fp32(1-0.999) by 1.3e-5 relative).
        assert np.all(np.abs(m - c * (1 - 0.9 ** t)) <= (1e-6 + 4 * t * EPS32) * np.abs(c))
        assert np.all(np.abs(v - c * c * (1 - 0.999 ** t)) <= 2e-5 * c * c)
        u_cf = (m_cf / bc1) / (np.sqrt(v_cf / bc2) + eps)
        assert np.all(np.abs(u_cf - c / (np.abs(c) + hp["eps"])) <= 1e-5)
        p_cf = p_cf - lr * u_cf
        assert np.all(np.abs(p - p_cf) <= t * (8 * EPS32 * (np.abs(p_cf) + hp["lr"]))), \
            f"p off at t={t}"


def pin_eps_placement(o):
    """eps is added outside the square root, after bias correction: with a
    dyadic c and eps = |c|, step 1 gives u = c/(|c|+|c|) = sign(c)/2 exactly."""
    world = 4
    c = np.array([2.0 ** -10, -(2.0 ** -10), 2.0 ** -10], np.float32)
    grads = [to_bf16_exact(c)] * world
    hp = dict(HP, eps=2.0 ** -10)
    p0 = np.array([0.5, -0.25, 0.0], np.float32)
    p, m, v = p0.copy(), np.zeros(3, np.float32), np.zeros(3, np.float32)
    one_rank_step(o, grads, p, m, v, 1, hp)
    decay = f32(1 - hp["lr"] * hp["wd"])
    expect = (p0 * decay - f32(hp["lr"]) * np.sign(c) * f32(0.5)).astype(np.float32)
    assert np.array_equal(p, expect), (p, expect)


def pin_lr0_wd0(o):
    """lr = 0 and wd = 0: the master is unchanged bit for bit; the moments
    still follow the gradient."""
    n, world = 777, 3
    grads = [synth.fill(n, seed=9, rank=j, step=1, bf16=True) for j in range(world)]
    master = synth.fill(n, seed=9, stream=synth.STREAM_MASTER, sigma=0.02)
    p, m, v = master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    one_rank_step(o, grads, p, m, v, 1, dict(HP, lr=0.0, wd=0.0))
    assert np.array_equal(p, master)
    assert np.count_nonzero(m) > n // 2


def pin_fp64_bound(o):
    """Against Adam carried out in float64 from the same fp32 coefficients and
    the exact mean gradient: every fp32 state stays within a first-order
    rounding-error bound propagated through the recurrences."""
    n, world, steps = 3000, 4, 12
    hp = HP
    master = synth.fill(n, seed=21, stream=synth.STREAM_MASTER, sigma=0.02)
    p, m, v = master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    P, M, V = master.astype(np.float64), np.zeros(n), np.zeros(n)
    dP, dM, dV = np.zeros(n), np.zeros(n), np.zeros(n)
    e = EPS32
    for t in range(1, steps + 1):
        grads = [synth.fill(n, seed=21, rank=j, step=t, bf16=True,
                            outlier_frac=0.05, outlier_scale=100.0) for j in range(world)]
        one_rank_step(o, grads, p, m, v, t, hp)
        sc = [float(x) for x in o.scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                                            hp["wd"], t, world)]
        b1, b2, omb1, omb2, bc1, bc2, lr, eps, decay, invN = sc
        xs = [bf16_to_f32(g).astype(np.float64) for g in grads]
        G = sum(xs) * invN
        dG = e * (world * sum(np.abs(x) for x in xs) * invN + np.abs(G))
        M_new = b1 * M + omb1 * G
        dM = b1 * dM + omb1 * dG + 3 * e * (b1 * np.abs(M) + omb1 * np.abs(G))
        V_new = b2 * V + omb2 * G * G
        dV = b2 * dV + omb2 * 2 * np.abs(G) * dG + 4 * e * (b2 * V + omb2 * G * G)
        M, V = M_new, V_new
        MH, VH = M / bc1, V / bc2
        dMH = dM / bc1 + e * np.abs(MH)
        dVH = dV / bc2 + e * VH
        SQ = np.sqrt(VH)
        dSQ = np.minimum(np.sqrt(dVH), dVH / np.maximum(SQ, 1e-300)) + e * SQ
        DEN = SQ + eps
        dDEN = dSQ + e * DEN
        U = MH / DEN
        dU = (dMH + np.abs(U) * dDEN) / np.maximum(DEN - dDEN, 1e-300) + e * np.abs(U)
        P_new = P * decay - lr * U
        dP = decay * dP + lr * dU + 2 * e * (np.abs(P) * decay + lr * np.abs(U))
        P = P_new
        for name, got, ref, bound in (("m", m, M, dM), ("v", v, V, dV), ("p", p, P, dP)):
            err = np.abs(got.astype(np.float64) - ref)
            assert np.all(err <= 2 * bound + 1e-45), \
                f"{name} exceeds the rounding bound at t={t}: {np.max(err / (2 * bound + 1e-45))}"


def pin_bias_correction_t2(o):
    """t = 2, constant dyadic c: bc1 = 1 - b1^2 and bc2 = 1 - b2^2 undo the
    moments' start-up bias: m_hat = c and v_hat = c^2 within a few ulp."""
    world = 2
    c = np.array([0.5, -0.125], np.float32)
    grads = [to_bf16_exact(c)] * world
    hp = dict(HP, wd=0.0, eps=0.0)
    p, m, v = np.zeros(2, np.float32), np.zeros(2, np.float32), np.zeros(2, np.float32)
    one_rank_step(o, grads, p, m, v, 1, hp)
    one_rank_step(o, grads, p, m, v, 2, hp)
    sc = o.scalars(hp["lr"], hp["beta1"], hp["beta2"], 0.0, 0.0, 2, world)
    assert abs(float(sc[4]) - 0.19) <= 0.19 * EPS32 * 2
    assert abs(float(sc[5]) - (1 - 0.999 ** 2)) <= (1 - 0.999 ** 2) * EPS32 * 2
    mh = m.astype(np.float64) / float(sc[4])
    vh = v.astype(np.float64) / float(sc[5])
    assert np.all(np.abs(mh - c) <= 8 * EPS32 * np.abs(c))
    assert np.all(np.abs(vh - c.astype(np.float64) ** 2) <= 8 * EPS32 * c.astype(np.float64) ** 2)
    # Two unit steps of lr in the direction -sign(c).
    assert np.all(np.abs(p + 2 * hp["lr"] * np.sign(c)) <= 16 * EPS32 * hp["lr"])


# ------------------------------------------------------------ O3 reduce ------
def _reduced_gradient(o, grads):
    """With beta1 = 0 (so 1-beta1 = 1), lr = wd = 0, step 1 leaves m = g exactly."""
    n = grads[0].size
    p, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    one_rank_step(o, grads, p, m, v, 1, dict(lr=0.0, beta1=0.0, beta2=0.999, eps=1e-8, wd=0.0))
    return m


def pin_reduce_dyadic(o):
    """Small dyadic inputs: the fp32 sum is exact, so the reduced gradient is
    the exact mean (N a power of two) — the data-parallel average gradient."""
    rng = np.random.default_rng(4)
    for world in (1, 2, 4, 8, 16):
        ints = rng.integers(-64, 65, size=(world, 257))
        vals = (ints * 2.0 ** -8).astype(np.float32)
        grads = [to_bf16_exact(vals[j]) for j in range(world)]
        g = _reduced_gradient(o, grads)
        exact = [Fraction(int(s), 256 * world) for s in ints.sum(axis=0)]
        assert all(Fraction(float(a)) == b for a, b in zip(g, exact)), f"N={world}"


def pin_reduce_order(o):
    """The slices are summed in ascending source-rank order: 1 + 2^24 rounds
    back to 2^24, then -2^24 cancels it, so the mean is 0 (descending order
    would give 1/4)."""
    vals = np.array([[1.0], [2.0 ** 24], [-(2.0 ** 24)], [0.0]], np.float32)
    grads = [to_bf16_exact(vals[j]) for j in range(4)]
    g = _reduced_gradient(o, grads)
    assert g[0] == 0.0


def pin_reduce_mean(o):
    """N identical slices give back the slice (mean, not sum), also for N not a
    power of two where 1/N is rounded: (x+x+x)*fp32(1/3) is x within 1 ulp."""
    x = synth.fill(500, seed=1, rank=0, step=1, bf16=True)
    xf = bf16_to_f32(x)
    for world in (2, 4, 8):
        assert np.array_equal(_reduced_gradient(o, [x] * world), xf)
    g3 = _reduced_gradient(o, [x] * 3)
    assert np.all(np.abs(g3 - xf) <= np.spacing(np.abs(xf)))
    # fp32 incoming slices are read as they are.
    xf32 = synth.fill(500, seed=2, rank=0, step=1)
    assert np.array_equal(_reduced_gradient(o, [xf32] * 4), xf32)


# -------------------------------------------------------------- O5 cast ------
def pin_cast_sampled(o):
    """bf16 and 3-byte rounding of fp32 against the exact-rational nearest
    value (ties to even), on special patterns and a random sample."""
    rng = np.random.default_rng(7)
    pats = special_float_patterns() + list(rng.integers(0, 2 ** 32, size=3000, dtype=np.uint64))
    xs = np.array(pats, dtype=np.uint32).view(np.float32)
    got16 = o.bf16(xs)
    for x, g in zip(xs, got16):
        ref = nearest_even_keep_high(x, 16)
        if ref is None:
            assert (int(g) & 0x7F80) == 0x7F80 and (int(g) & 0x7F) != 0
        else:
            assert int(g) == ref, (hex(int(np.array(x).view(np.uint32))), hex(int(g)), hex(ref))
        ref24 = nearest_even_keep_high(x, 8)
        g24 = o.fp24(x)
        if ref24 is None:
            assert (g24 & 0x7F8000) == 0x7F8000 and (g24 & 0x7FFF) != 0
        else:
            assert g24 == ref24, (hex(int(np.array(x).view(np.uint32))), hex(g24), hex(ref24))


def pin_cast_ranges(o):
    """The range casts (the expected values of the GPU's exhaustive cast test)
    are the pinned element casts of the patterns first, first + 1, ... (mod
    2^32), the 3-byte one stored little-endian: windows around every boundary
    of both formats, random windows, and one that wraps past 0xFFFFFFFF."""
    rng = np.random.default_rng(5)
    starts = [0, 0x7F - 40, 0x00800000 - 300, 0x7F7FFF00 - 200, 0x7F800000 - 300,
              0x7FFFFFFF - 100, 0x80000000 - 20, 0xFF7FFF00, 0xFFFFFFFF - 150]
    starts += [int(x) for x in rng.integers(0, 1 << 32, size=12)]
    # windows across bf16 rounding ties (low 16 bits 0x8000), where a pattern
    # and its neighbour round differently
    starts += [(int(k) << 16) + 0x8000 - 150 for k in rng.integers(0, 1 << 16, size=6)]
    n = 400
    for first in starts:
        pats = (np.arange(first, first + n, dtype=np.uint64) % (1 << 32)).astype(np.uint32)
        assert np.array_equal(o.bf16_bits_range(first, n), o.bf16(pats.view(np.float32))), \
            hex(first)
        b = o.fp24_bits_range(first, n).reshape(n, 3).astype(np.uint32)
        packed = b[:, 0] | (b[:, 1] << 8) | (b[:, 2] << 16)
        for i in range(n):
            x = pats[i:i + 1].view(np.float32)[0]
            assert int(packed[i]) == o.fp24(x), hex(int(pats[i]))


def pin_param_store(o):
    """The parameter written into the slot is the nearest-even rounding of the
    updated fp32 master: bf16 (2 B), 3-byte (little-endian) or an fp32 copy."""
    n, world = 333, 2
    grads = [synth.fill(n, seed=8, rank=j, step=1, bf16=True) for j in range(world)]
    master = synth.fill(n, seed=8, stream=synth.STREAM_MASTER, sigma=0.02)
    for dt in (orc.BF16, orc.FP24, orc.FP32):
        p, m, v = master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        out = one_rank_step(o, grads, p, m, v, 1, param_dtype=dt)
        if dt == orc.FP32:
            assert np.array_equal(out.view(np.float32), p)
            continue
        if dt == orc.BF16:
            got = out.view(np.uint16).astype(np.int64)
        else:
            b = out.reshape(n, 3).astype(np.int64)
            got = b[:, 0] | (b[:, 1] << 8) | (b[:, 2] << 16)
        drop = 16 if dt == orc.BF16 else 8
        for k in range(0, n, 7):
            assert got[k] == nearest_even_keep_high(p[k], drop)


# -------------------------------------------------------------- O1 plan ------
def pin_plan_bruteforce(o):
    """All tiny parameter lists (up to 3 tensors of 1..4 elements, every tie
    pattern), N in 1..4, align in {1, 2, 4}: unique tensors are laid out
    back to back in registration order, ties alias their owner, P_pad is the
    least multiple of N*align >= P, shards tile [0, P_pad), and the round trip
    flatten -> shard -> gather -> unflatten is the identity on random bits."""
    rng = np.random.default_rng(0)
    for k in range(0, 4):
        for numels in itertools.product(range(1, 5), repeat=k):
            tie_choices = [[-1]] + [[-1] + list(range(i)) for i in range(1, k)]
            for ties in itertools.product(*tie_choices[:k]):
                ties = list(ties)
                root = []
                for i, t in enumerate(ties):
                    root.append(i if t < 0 else root[t])
                if any(numels[root[i]] != numels[i] for i in range(k)):
                    continue
                for world in range(1, 5):
                    for align in (1, 2, 4):
                        _check_plan_case(o, list(numels), ties, root, world, align, rng)


def _check_plan_case(o, numels, ties, root, world, align, rng):
    plan = o.plan(numels, ties, world=world, align=align)
    P = sum(n for i, n in enumerate(numels) if root[i] == i)
    assert plan["P"] == P
    Q = world * align
    assert plan["P_pad"] % Q == 0 and plan["P_pad"] >= P and plan["P_pad"] - P < Q
    S = plan["S"]
    assert S * world == plan["P_pad"]
    expect_off, cur = [], 0
    for i, n in enumerate(numels):
        if root[i] == i:
            expect_off.append(cur)
            cur += n
        else:
            expect_off.append(expect_off[root[i]])
    assert list(plan["offsets"]) == expect_off
    # Shard ranges of the whole buffer tile [0, P_pad) in rank order.
    covered = []
    for r in range(world):
        lo, hi = o.shard_range(0, plan["P_pad"], r, S)
        assert (lo, hi) == (0, S)
        covered += list(range(r * S + lo, r * S + hi))
    assert covered == list(range(plan["P_pad"]))
    # Round trip on random 16-bit patterns (NaN payloads included).
    tensors = [rng.integers(0, 2 ** 16, size=n, dtype=np.uint16) for n in numels]
    flat = np.zeros(plan["P_pad"], np.uint16)
    for i, n in enumerate(numels):
        if root[i] == i:
            flat[expect_off[i]: expect_off[i] + n] = tensors[i]
    shards = [flat[j * S:(j + 1) * S].copy() for j in range(world)]
    out = np.full(plan["P_pad"] + 4, 0xABCD, np.uint16)
    o.gather(world=world, S=S, elem_size=2, shards=shards, full_flat=out)
    assert np.all(out[plan["P_pad"]:] == 0xABCD), "gather wrote past the buffer"
    for i, n in enumerate(numels):
        off = plan["offsets"][i]
        assert np.array_equal(out[off:off + n], tensors[root[i]])
    assert not out[P:plan["P_pad"]].any(), "pad is not zero"


def pin_plan_buckets(o):
    """Buckets over random lists: contiguous, newest-first, covering [0, P_pad)
    with the pad in the first; whole tensors only; each bucket within B unless
    it is one oversized tensor; greedy: the next tensor would overflow it."""
    rng = np.random.default_rng(1)
    for case in range(400):
        k = int(rng.integers(1, 9))
        numels = [int(x) for x in rng.integers(1, 40, size=k)]
        B = int(rng.integers(1, 80))
        world = int(rng.integers(1, 5))
        plan = o.plan(numels, None, world=world, align=2, bucket_elems=B)
        offs = plan["offsets"]
        bks = plan["buckets"]
        assert bks[0][1] == plan["P_pad"] and bks[-1][0] == 0
        for a, b in zip(bks, bks[1:]):
            assert b[1] == a[0]
        starts = {int(x) for x in offs}
        idx_of_start = {int(offs[i]): i for i in range(k)}
        for bi, (lo, hi) in enumerate(bks):
            assert lo in starts
            members = [i for i in range(k) if lo <= offs[i] < min(hi, plan["P"])]
            size = sum(numels[i] for i in members)
            assert size <= B or len(members) == 1
            if bi + 1 < len(bks):
                nxt = idx_of_start[lo] - 1
                assert nxt >= 0 and size + numels[nxt] > B, "bucket not greedy"


def pin_plan_workloads(o):
    """P of the four model-shaped lists against the architectures' closed-form
    parameter counts, and the tie handling (a tied head adds nothing)."""
    def gpt2(V, npos, L, d, ffn):
        return V * d + npos * d + L * (4 * d * d + 2 * d * ffn + 9 * d + ffn) + 2 * d

    def qwen2(V, L, d, ffn, q, kv):
        return V * d + L * (2 * d + q * d + q + 2 * (kv * d + kv) + d * q + 3 * d * ffn) + d

    def llama(V, L, d, ffn):
        return 2 * V * d + L * (2 * d + 4 * d * d + 3 * d * ffn) + d

    expect = {TINY.key: gpt2(1000, 0, 2, 256, 1024),
              GPT2_SMALL.key: gpt2(50257, 1024, 12, 768, 3072),
              QWEN25_3B.key: qwen2(151936, 36, 2048, 11008, 2048, 256),
              LLAMA_7B.key: llama(32000, 32, 4096, 11008)}
    approx = {GPT2_SMALL.key: 124e6, QWEN25_3B.key: 3.09e9, LLAMA_7B.key: 6.7e9}
    for w in (TINY, GPT2_SMALL, QWEN25_3B, LLAMA_7B):
        plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align,
                      bucket_elems=w.bucket_elems)
        assert plan["P"] == expect[w.key], w.key
        if w.key in approx:
            assert abs(plan["P"] - approx[w.key]) / approx[w.key] < 0.006
        Q = w.world * w.align
        assert plan["P_pad"] == -(-plan["P"] // Q) * Q
        for i, p in enumerate(w.params):
            if p.tied_to >= 0:
                assert plan["offsets"][i] == plan["offsets"][p.tied_to]


# ------------------------------------------------------------ O2 ledger ------
def read_golden_ledger():
    rows = {}
    with open(os.path.join(GOLDEN, "ledger_pages.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val, kind, _cite = [c.strip() for c in line.split("|", 3)]
            rows[key] = (float(val), kind)
    return rows


def pin_ledger_pages(o):
    """The per-rank ledger against the numbers the pages print, and the kept
    buffers against the pages' per-stage formulas, exactly, in integers."""
    g = read_golden_ledger()

    def check(key, got):
        val, kind = g[key]
        tol = 1e-9 * max(1.0, abs(val)) if kind == "exact" else (1.0 if val > 5 else 0.05)
        assert abs(got - val) <= tol, (key, got, val)

    bpp = o.ledger_bytes_per_param
    check("ddp_bytes_per_param", bpp(0, 8))
    check("dp2zero_ddp_per_param", bpp(0, 8))
    check("ddp_7B_GB", 7e9 * bpp(0, 8) / 1e9)
    check("lifecycle_7B_GB", 7e9 * bpp(0, 8) / 1e9)
    check("dp2zero_7B_GB", 7e9 * bpp(0, 8) / 1e9)
    check("ddp_70B_TB", 70e9 * bpp(0, 8) / 1e12)
    # Optimizer bytes are the part ZeRO-1 divides by N: 2 * (Z1(1) - Z1(2)) = 12.
    check("optimizer_share", 2 * (bpp(1, 1) - bpp(1, 2)) / bpp(0, 1))
    check("zero1_dp8_opt_bytes", bpp(1, 8) - 4)
    check("zero1_dp8_bytes_per_param", bpp(1, 8))
    check("zero1_dp8_7B_GB", 7e9 * bpp(1, 8) / 1e9)
    check("zero2_dp8_bytes_per_param", bpp(2, 8))
    check("zero2_dp8_7B_GB", 7e9 * bpp(2, 8) / 1e9)
    check("zero3_dp8_bytes_per_param", bpp(3, 8))
    check("zero3_dp8_7B_GB", 7e9 * bpp(3, 8) / 1e9)
    check("lifecycle_zero3_per_param", bpp(3, 8) * 8)
    # The 70B ZeRO-3 figures: the page's own formula gives 140 GB per rank;
    # its per-card 17.5 GB is the bf16 parameter shard alone.
    assert abs(70e9 * bpp(3, 8) / 1e9 - 140.0) < 1e-9
    check("zero3_dp8_70B_params_GB", 70e9 * 2 / 8 / 1e9)
    plan = o.plan(QWEN25_3B.numels, QWEN25_3B.tied_to, world=4)
    for stage, key in ((1, "qwen3b_n4_zero1_GB"), (2, "qwen3b_n4_zero2_GB"),
                       (3, "qwen3b_n4_zero3_GB")):
        check(key, o.ledger_kept_bytes(stage, plan["P_pad"], 4) / 1e9)
    # Kept buffers == formula, exactly, for every stage and N.
    for world in (1, 2, 3, 4, 8, 64):
        P_pad = world * 128 * 1001
        for stage in (0, 1, 2, 3):
            kept = o.ledger_kept_bytes(stage, P_pad, world)
            per = Fraction(o.ledger_bytes_per_param(stage, world)).limit_denominator(1000)
            assert Fraction(kept) == per * P_pad, (stage, world)


# ------------------------------------------------------ O6/O7 equivalence ----
def _local_grads(w, P_pad, P, t, n_ranks):
    return [synth.fill(P_pad, seed=w.seed, rank=j, step=t, sigma=w.grad_sigma, p_limit=P,
                       outlier_frac=w.outlier_frac, outlier_scale=w.outlier_scale, bf16=True)
            for j in range(n_ranks)]


def pin_ddp_equivalence(o, w=TINY, steps=None):
    """The N shard-local steps, concatenated and all-gathered, equal the
    unsharded DDP AllReduce + AdamW step bit for bit, for every step."""
    plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align)
    P, P_pad, S, N = plan["P"], plan["P_pad"], plan["S"], w.world
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    ddp = dict(master=master0.copy(), m=np.zeros(P_pad, np.float32),
               v=np.zeros(P_pad, np.float32), params=np.zeros(P_pad, np.uint16))
    sh_master = [master0[r * S:(r + 1) * S].copy() for r in range(N)]
    sh_m = [np.zeros(S, np.float32) for _ in range(N)]
    sh_v = [np.zeros(S, np.float32) for _ in range(N)]
    hp = w.hparams
    hp = dict(lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
              wd=hp["weight_decay"])
    for t in range(1, (steps or w.steps) + 1):
        local = _local_grads(w, P_pad, P, t, N)
        o.ddp_step(world=N, P_pad=P_pad, local_grads=local, **ddp, t=t, **hp)
        fulls = []
        for r in range(N):
            full = np.zeros(P_pad, np.uint16)
            slices = [local[j][r * S:(r + 1) * S].copy() for j in range(N)]
            o.shard_step(world=N, rank=r, S=S, lo=0, hi=S, grads=slices, master=sh_master[r],
                         m=sh_m[r], v=sh_v[r], full_flat=full, t=t, **hp)
            fulls.append(full)
        own = [fulls[r][r * S:(r + 1) * S].copy() for r in range(N)]
        gathered = np.zeros(P_pad, np.uint16)
        o.gather(world=N, S=S, elem_size=2, shards=own, full_flat=gathered)
        assert np.array_equal(gathered, ddp["params"]), f"params differ at t={t}"
        for name, shards in (("master", sh_master), ("m", sh_m), ("v", sh_v)):
            assert np.array_equal(np.concatenate(shards).view(np.uint32),
                                  ddp[name].view(np.uint32)), f"{name} differs at t={t}"
        assert not gathered[P:].any() and not ddp["master"][P:].any()


def pin_ddp_equivalence_gpt2_buckets(o, steps=1):
    """The C2 configuration at full size: the GPT-2-small list over N = 8
    ranks with 25M-element buckets, each rank's step run bucket by bucket (its
    shard-local part of every bucket), gathered, equals the unsharded DDP
    AllReduce + AdamW step bit for bit (parameters, master, m, v), and the
    768-element tail pad stays zero."""
    w = GPT2_SMALL
    plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align,
                  bucket_elems=w.bucket_elems)
    P, P_pad, S, N = plan["P"], plan["P_pad"], plan["S"], w.world
    assert len(plan["buckets"]) == 5 and P_pad - P == 768
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    ddp = dict(master=master0.copy(), m=np.zeros(P_pad, np.float32),
               v=np.zeros(P_pad, np.float32), params=np.zeros(P_pad, np.uint16))
    sh = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
          for r in range(N)]
    hp = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, wd=w.weight_decay)
    for t in range(1, steps + 1):
        local = _local_grads(w, P_pad, P, t, N)
        o.ddp_step(world=N, P_pad=P_pad, local_grads=local, **ddp, t=t, **hp)
        own = []
        for r in range(N):
            full = np.zeros(P_pad, np.uint16)
            slices = [local[j][r * S:(r + 1) * S].copy() for j in range(N)]
            for flo, fhi in plan["buckets"]:
                lo, hi = o.shard_range(flo, fhi, r, S)
                if lo < hi:
                    o.shard_step(world=N, rank=r, S=S, lo=lo, hi=hi, grads=slices,
                                 master=sh[r][0], m=sh[r][1], v=sh[r][2], full_flat=full, t=t,
                                 **hp)
            own.append(full[r * S:(r + 1) * S].copy())
        gathered = np.zeros(P_pad, np.uint16)
        o.gather(world=N, S=S, elem_size=2, shards=own, full_flat=gathered)
        assert np.array_equal(gathered, ddp["params"]), f"params differ at t={t}"
        for k, name in enumerate(("master", "m", "v")):
            assert np.array_equal(np.concatenate([x[k] for x in sh]).view(np.uint32),
                                  ddp[name].view(np.uint32)), f"{name} differs at t={t}"
        assert not gathered[P:].any() and not ddp["master"][P:].any()


def pin_bucket_invariance(o):
    """A step run as per-bucket sub-range calls equals the whole-shard call bit
    for bit (the step is element-local)."""
    params = gpt2_params(2, 64, 256, 500, 32)
    numels = [p.numel for p in params]
    ties = [p.tied_to for p in params]
    N = 4
    plan = o.plan(numels, ties, world=N, align=128, bucket_elems=20000)
    assert len(plan["buckets"]) >= 4
    P, P_pad, S = plan["P"], plan["P_pad"], plan["S"]
    master0 = synth.fill(P_pad, seed=2, stream=synth.STREAM_MASTER, sigma=0.02, p_limit=P)
    for r in range(N):
        whole = [master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
        parts = [a.copy() for a in whole]
        fw = np.zeros(P_pad, np.uint16)
        fp = np.zeros(P_pad, np.uint16)
        for t in (1, 2):
            sl = [synth.fill(S, index0=r * S, seed=2, rank=j, step=t, p_limit=P, bf16=True)
                  for j in range(N)]
            o.shard_step(world=N, rank=r, S=S, lo=0, hi=S, grads=sl, master=whole[0],
                         m=whole[1], v=whole[2], full_flat=fw, t=t, **HP)
            for (flo, fhi) in plan["buckets"]:
                lo, hi = o.shard_range(flo, fhi, r, S)
                if hi > lo:
                    o.shard_step(world=N, rank=r, S=S, lo=lo, hi=hi, grads=sl,
                                 master=parts[0], m=parts[1], v=parts[2], full_flat=fp, t=t,
                                 **HP)
            for a, b in zip(whole, parts):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
            assert np.array_equal(fw, fp)


# --------------------------------------------------- global-norm clipping ----
def pin_sqnorm_dyadic(o):
    """Small dyadic slices: the sum of squares of the mean gradient is exact in
    double, equal to the rational closed form."""
    rng = np.random.default_rng(12)
    for world in (1, 2, 4, 8):
        ints = rng.integers(-64, 65, size=(world, 333))
        vals = (ints * 2.0 ** -8).astype(np.float32)
        grads = [to_bf16_exact(vals[j]) for j in range(world)]
        got = o.grad_sqnorm(world=world, S=333, lo=0, hi=333, grads=grads)
        exact = sum(Fraction(int(x), 256 * world) ** 2 for x in ints.sum(axis=0))
        assert Fraction(got) == exact, world
        lo, hi = 17, 300
        part = o.grad_sqnorm(world=world, S=333, lo=lo, hi=hi, grads=grads)
        assert Fraction(part) == sum(Fraction(int(x), 256 * world) ** 2
                                     for x in ints.sum(axis=0)[lo:hi])


def pin_clip_coef_closed_forms(o):
    """min(1, max_norm / (norm + 1e-6)) in fp32; the partial sums add in rank
    order; an infinite or NaN norm sets the shared skip flag."""
    c, bad = o.clip_coef([9.0, 16.0], 1.0)
    assert bad == 0 and c == np.float32(1.0 / (5.0 + 1e-6))
    c, bad = o.clip_coef([9.0, 16.0], 100.0)
    assert bad == 0 and c == np.float32(1.0)
    c, bad = o.clip_coef([4.0, 0.0, 0.0], 1.0)
    assert bad == 0 and c == np.float32(1.0 / (2.0 + 1e-6))
    c, bad = o.clip_coef([0.0], 1.0)
    assert bad == 0 and c == np.float32(1.0)
    for rank_sq in ([float("inf"), 1.0], [1.0, float("nan")], [1e308, 1e308]):
        c, bad = o.clip_coef(rank_sq, 1.0)
        assert bad == 1 and c == np.float32(1.0), rank_sq
    c, bad = o.clip_coef([1e300, 1e300], 1.0)
    assert bad == 0 and c == np.float32(1.0 / (np.sqrt(2e300) + 1e-6))


def _clip_inputs(n=2048, world=4, seed=31):
    grads = [synth.fill(n, seed=seed, rank=j, step=1, bf16=True, outlier_frac=0.02,
                        outlier_scale=50.0) for j in range(world)]
    master = synth.fill(n, seed=seed, stream=synth.STREAM_MASTER, sigma=0.02)
    return grads, master


def pin_clip_unit_identity(o):
    """coef = 1 and no skip is the unclipped step, bit for bit."""
    grads, master = _clip_inputs()
    n, world = master.size, len(grads)
    a = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    fa = np.zeros(n * world, np.uint16)
    fb = np.zeros(n * world, np.uint16)
    for t in (1, 2):
        o.shard_step(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=a[0], m=a[1],
                     v=a[2], full_flat=fa, t=t, **HP)
        o.shard_step_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=b[0],
                             m=b[1], v=b[2], full_flat=fb, coef=1.0, skip=0, t=t, **HP)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert np.array_equal(fa, fb)


def pin_clip_post_norm(o):
    """After clipping to max_norm, the gradient the update sees has global
    norm max_norm * norm / (norm + 1e-6) (observed as m with beta1 = 0)."""
    grads, master = _clip_inputs()
    n, world = master.size, len(grads)
    sq = o.grad_sqnorm(world=world, S=n, lo=0, hi=n, grads=grads)
    norm = np.sqrt(sq)
    max_norm = 0.25 * norm
    coef, bad = o.clip_coef([sq], max_norm)
    assert bad == 0 and coef < 1
    m = np.zeros(n, np.float32)
    o.shard_step_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=master.copy(),
                         m=m, v=np.zeros(n, np.float32), full_flat=np.zeros(n * world, np.uint16),
                         coef=coef, skip=0, t=1, lr=0.0, beta1=0.0, beta2=0.999, eps=1e-8,
                         wd=0.0)
    got = np.sqrt(np.sum(m.astype(np.float64) ** 2))
    expect = max_norm * norm / (norm + 1e-6)
    assert abs(got - expect) <= 4e-7 * expect, (got, expect)


def pin_clip_skip(o):
    """A skipped step leaves master, m, v and the parameter slot untouched."""
    grads, master = _clip_inputs()
    n, world = master.size, len(grads)
    st = [master.copy(), np.full(n, 0.5, np.float32), np.full(n, 0.25, np.float32)]
    full = np.full(n * world, 0x1234, np.uint16)
    before = [x.copy() for x in st] + [full.copy()]
    o.shard_step_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=st[0],
                         m=st[1], v=st[2], full_flat=full, coef=0.5, skip=1, t=3, **HP)
    for x, y in zip(st + [full], before):
        assert np.array_equal(x, y)


def pin_clip_ddp_equivalence(o, w=TINY, steps=2):
    """Clipping on the global norm: the sharded pipeline (each rank's partial
    sum of squares, the coefficient over the N partials, N clipped shard steps,
    gather) equals the unsharded clipped step over the whole flat buffer, bit
    for bit, and both see the same coefficient."""
    plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align)
    P, P_pad, S, N = plan["P"], plan["P_pad"], plan["S"], w.world
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    full_st = [master0.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    full_params = np.zeros(P_pad * N, np.uint16)   # rank-0 "slot" spans the whole buffer
    sh = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
          for r in range(N)]
    max_norm = None
    for t in range(1, steps + 1):
        local = _local_grads(w, P_pad, P, t, N)
        sq_full = o.grad_sqnorm(world=N, S=P_pad, lo=0, hi=P_pad, grads=local)
        if max_norm is None:
            max_norm = 0.5 * float(np.sqrt(sq_full))
        c_full, bad_full = o.clip_coef([sq_full], max_norm)
        o.shard_step_clipped(world=N, rank=0, S=P_pad, lo=0, hi=P_pad, grads=local,
                             master=full_st[0], m=full_st[1], v=full_st[2], full_flat=full_params,
                             coef=c_full, skip=bad_full, t=t, **HP)
        slices = [[local[j][r * S:(r + 1) * S].copy() for j in range(N)] for r in range(N)]
        partial = [o.grad_sqnorm(world=N, S=S, lo=0, hi=S, grads=slices[r]) for r in range(N)]
        c_sh, bad_sh = o.clip_coef(partial, max_norm)
        assert bad_sh == bad_full == 0 and c_sh == c_full and c_sh < 1, (c_sh, c_full)
        fulls = []
        for r in range(N):
            f = np.zeros(P_pad, np.uint16)
            o.shard_step_clipped(world=N, rank=r, S=S, lo=0, hi=S, grads=slices[r],
                                 master=sh[r][0], m=sh[r][1], v=sh[r][2], full_flat=f,
                                 coef=c_sh, skip=bad_sh, t=t, **HP)
            fulls.append(f[r * S:(r + 1) * S].copy())
        gathered = np.zeros(P_pad, np.uint16)
        o.gather(world=N, S=S, elem_size=2, shards=fulls, full_flat=gathered)
        assert np.array_equal(gathered, full_params[:P_pad]), f"params differ at t={t}"
        for k in range(3):
            assert np.array_equal(np.concatenate([x[k] for x in sh]).view(np.uint32),
                                  full_st[k].view(np.uint32)), f"state {k} differs at t={t}"


# ------------------------------------------------- gradient accumulation ----
def _accum_run(o, micro, world, S, master, hp=HP, t=1, stale=None):
    """Run G = len(micro) micro-steps (each a list of N slices) through the
    accumulator and the accumulated step; return (master, m, v, params)."""
    G = len(micro)
    acc = np.full(S, np.nan, np.float32) if stale is None else stale.copy()
    for k in range(G - 1):
        o.grad_accumulate(world=world, S=S, lo=0, hi=S, grads=micro[k], accum=acc, first=k == 0)
    if G == 1:
        acc = np.zeros(S, np.float32)
    st = [master.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    full = np.zeros(S * world, np.uint16)
    o.shard_step_accumulated(world=world, rank=0, S=S, lo=0, hi=S, grads=micro[G - 1],
                             accum=acc, micro_steps=G, master=st[0], m=st[1], v=st[2],
                             full_flat=full, t=t, **hp)
    return st + [full]


def pin_accum_single_microstep_identity(o):
    """G = 1 with a zero accumulator is the plain step, bit for bit."""
    grads, master = _clip_inputs(n=1500, world=4, seed=41)
    a = _accum_run(o, [grads], 4, 1500, master)
    b = [master.copy(), np.zeros(1500, np.float32), np.zeros(1500, np.float32)]
    fb = np.zeros(1500 * 4, np.uint16)
    o.shard_step(world=4, rank=0, S=1500, lo=0, hi=1500, grads=grads, master=b[0], m=b[1],
                 v=b[2], full_flat=fb, t=1, **HP)
    for x, y in zip(a, b + [fb]):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def pin_accum_dyadic(o):
    """Dyadic micro-batches: the gradient the update sees is the exact average
    over the G micro-batches and the N ranks (exact for G a power of two,
    within one fp32 rounding of the exact value otherwise); observed as m with
    beta1 = 0."""
    rng = np.random.default_rng(8)
    world, S = 4, 257
    for G in (2, 3, 4, 5, 8):
        ints = rng.integers(-32, 33, size=(G, world, S))
        micro = [[to_bf16_exact((ints[k, j] * 2.0 ** -8).astype(np.float32)) for j in range(world)]
                 for k in range(G)]
        st = _accum_run(o, micro, world, S, np.zeros(S, np.float32),
                        hp=dict(lr=0.0, beta1=0.0, beta2=0.999, eps=1e-8, wd=0.0))
        g = st[1]
        exact = [Fraction(int(x), 256 * world * G) for x in ints.sum(axis=(0, 1))]
        for got, ex in zip(g, exact):
            if G & (G - 1) == 0:
                assert Fraction(float(got)) == ex, G
            else:
                ulp = abs(float(np.spacing(np.float32(float(ex)))))
                assert abs(Fraction(float(got)) - ex) <= Fraction(ulp), G


def pin_accum_equals_merged(o):
    """G = 2 micro-batches of N = 2 slices, dyadic: the same update as one step
    over the 4 slices together (the mean over micro-batches and ranks)."""
    rng = np.random.default_rng(9)
    S = 300
    ints = rng.integers(-16, 17, size=(4, S))
    sl = [to_bf16_exact((ints[j] * 2.0 ** -6).astype(np.float32)) for j in range(4)]
    master = synth.fill(S, seed=9, stream=synth.STREAM_MASTER, sigma=0.02)
    a = _accum_run(o, [sl[:2], sl[2:]], 2, S, master)
    b = [master.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
    fb = np.zeros(S * 4, np.uint16)
    o.shard_step(world=4, rank=0, S=S, lo=0, hi=S, grads=sl, master=b[0], m=b[1], v=b[2],
                 full_flat=fb, t=1, **HP)
    for x, y in zip(a[:3], b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert np.array_equal(a[3][:S], fb[:S])


def pin_accum_first_overwrites(o):
    """The first micro-step overwrites the accumulator: stale contents (NaN,
    leftovers of the previous optimizer step) never reach the update."""
    grads, master = _clip_inputs(n=800, world=2, seed=43)
    g2, _ = _clip_inputs(n=800, world=2, seed=44)
    clean = _accum_run(o, [grads, g2], 2, 800, master, stale=np.zeros(800, np.float32))
    dirty = _accum_run(o, [grads, g2], 2, 800, master, stale=np.full(800, np.nan, np.float32))
    for x, y in zip(clean, dirty):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert np.isfinite(clean[0]).all()


def pin_accum_ddp_equivalence(o, w=TINY, G=3, steps=2):
    """G micro-steps per optimizer step: the N ranks' accumulators and steps,
    gathered, equal the unsharded accumulation and step over the whole flat
    buffer, bit for bit."""
    plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align)
    P, P_pad, S, N = plan["P"], plan["P_pad"], plan["S"], w.world
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    full_st = [master0.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    full_acc = np.zeros(P_pad, np.float32)
    full_params = np.zeros(P_pad * N, np.uint16)
    sh = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
          for r in range(N)]
    sh_acc = [np.zeros(S, np.float32) for _ in range(N)]
    for t in range(1, steps + 1):
        for k in range(G):
            local = [synth.fill(P_pad, seed=w.seed, rank=j, step=1000 * t + k, sigma=w.grad_sigma,
                                p_limit=P, bf16=True) for j in range(N)]
            slices = [[local[j][r * S:(r + 1) * S].copy() for j in range(N)] for r in range(N)]
            if k < G - 1:
                o.grad_accumulate(world=N, S=P_pad, lo=0, hi=P_pad, grads=local, accum=full_acc,
                                  first=k == 0)
                for r in range(N):
                    o.grad_accumulate(world=N, S=S, lo=0, hi=S, grads=slices[r], accum=sh_acc[r],
                                      first=k == 0)
                continue
            o.shard_step_accumulated(world=N, rank=0, S=P_pad, lo=0, hi=P_pad, grads=local,
                                     accum=full_acc, micro_steps=G, master=full_st[0],
                                     m=full_st[1], v=full_st[2], full_flat=full_params, t=t, **HP)
            fulls = []
            for r in range(N):
                f = np.zeros(P_pad, np.uint16)
                o.shard_step_accumulated(world=N, rank=r, S=S, lo=0, hi=S, grads=slices[r],
                                         accum=sh_acc[r], micro_steps=G, master=sh[r][0],
                                         m=sh[r][1], v=sh[r][2], full_flat=f, t=t, **HP)
                fulls.append(f[r * S:(r + 1) * S].copy())
            gathered = np.zeros(P_pad, np.uint16)
            o.gather(world=N, S=S, elem_size=2, shards=fulls, full_flat=gathered)
            assert np.array_equal(gathered, full_params[:P_pad]), f"params differ at t={t}"
            for i in range(3):
                assert np.array_equal(np.concatenate([x[i] for x in sh]).view(np.uint32),
                                      full_st[i].view(np.uint32)), f"state {i} differs at t={t}"


# ------------------------------------------ clipping an accumulated step ----
def pin_accum_clip_reductions(o):
    """Clipping an accumulated gradient reduces to the pieces it is made of:
    G = 1 with a zero accumulator is the clipped step (norm and update, bit for
    bit); a coefficient of 1 without skip is the accumulated step; a skip
    leaves every buffer untouched."""
    grads, master = _clip_inputs(n=1700, world=4, seed=53)
    n, world = master.size, len(grads)
    zero = np.zeros(n, np.float32)
    assert o.grad_sqnorm_accumulated(world=world, S=n, lo=0, hi=n, grads=grads, accum=zero,
                                     micro_steps=1) == o.grad_sqnorm(world=world, S=n, lo=0,
                                                                     hi=n, grads=grads)
    for coef in (np.float32(0.3125), np.float32(0.7)):
        a = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
             np.zeros(n * world, np.uint16)]
        b = [x.copy() for x in a]
        o.shard_step_accumulated_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads,
                                         accum=zero, micro_steps=1, master=a[0], m=a[1], v=a[2],
                                         full_flat=a[3], coef=coef, skip=0, t=2, **HP)
        o.shard_step_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads, master=b[0],
                             m=b[1], v=b[2], full_flat=b[3], coef=coef, skip=0, t=2, **HP)
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    rng = np.random.default_rng(54)
    acc = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    a = [master.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
         np.zeros(n * world, np.uint16)]
    b = [x.copy() for x in a]
    o.shard_step_accumulated_clipped(world=world, rank=1, S=n, lo=5, hi=n - 3, grads=grads,
                                     accum=acc, micro_steps=3, master=a[0], m=a[1], v=a[2],
                                     full_flat=a[3], coef=1.0, skip=0, t=4, **HP)
    o.shard_step_accumulated(world=world, rank=1, S=n, lo=5, hi=n - 3, grads=grads, accum=acc,
                             micro_steps=3, master=b[0], m=b[1], v=b[2], full_flat=b[3], t=4,
                             **HP)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    before = [x.copy() for x in a]
    o.shard_step_accumulated_clipped(world=world, rank=1, S=n, lo=0, hi=n, grads=grads,
                                     accum=acc, micro_steps=3, master=a[0], m=a[1], v=a[2],
                                     full_flat=a[3], coef=0.5, skip=1, t=5, **HP)
    for x, y in zip(a, before):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def pin_accum_clip_dyadic(o):
    """Dyadic slices and accumulator, G and N powers of two: the accumulated
    norm is the exact rational sum of ((a + mean) / G)^2 over the range, and
    after clipping the update sees a gradient of norm
    max_norm * norm / (norm + 1e-6) (observed as m with beta1 = 0)."""
    rng = np.random.default_rng(55)
    n = 777
    for world, G in ((1, 2), (2, 4), (4, 2), (8, 8)):
        ints = rng.integers(-64, 65, size=(world, n))
        grads = [to_bf16_exact((ints[j] * 2.0 ** -8).astype(np.float32)) for j in range(world)]
        a_int = rng.integers(-512, 513, size=n)
        acc = (a_int * 2.0 ** -10).astype(np.float32)
        want = [(Fraction(int(a_int[i]), 1024) + Fraction(int(x), 256 * world)) / G
                for i, x in enumerate(ints.sum(axis=0))]
        got = o.grad_sqnorm_accumulated(world=world, S=n, lo=0, hi=n, grads=grads, accum=acc,
                                        micro_steps=G)
        assert Fraction(got) == sum(q * q for q in want), (world, G)
        lo, hi = 31, 700
        part = o.grad_sqnorm_accumulated(world=world, S=n, lo=lo, hi=hi, grads=grads, accum=acc,
                                         micro_steps=G)
        assert Fraction(part) == sum(q * q for q in want[lo:hi]), (world, G)
        norm = float(np.sqrt(got))
        max_norm = 0.375 * norm
        coef, bad = o.clip_coef([got], max_norm)
        assert bad == 0 and coef < 1
        m = np.zeros(n, np.float32)
        o.shard_step_accumulated_clipped(world=world, rank=0, S=n, lo=0, hi=n, grads=grads,
                                         accum=acc, micro_steps=G,
                                         master=np.zeros(n, np.float32), m=m,
                                         v=np.zeros(n, np.float32),
                                         full_flat=np.zeros(n * world, np.uint16), coef=coef,
                                         skip=0, t=1, lr=0.0, beta1=0.0, beta2=0.999, eps=1e-8,
                                         wd=0.0)
        seen = np.sqrt(np.sum(m.astype(np.float64) ** 2))
        expect = max_norm * norm / (norm + 1e-6)
        assert abs(seen - expect) <= 4e-7 * expect, (world, G, seen, expect)


def pin_accum_clip_ddp_equivalence(o, w=TINY, G=3, steps=2):
    """G micro-steps and global-norm clipping of their average: the sharded
    pipeline (N accumulators, each rank's partial norm of its accumulated
    gradient, the coefficient over the N partials, N clipped accumulated steps,
    gather) equals the unsharded one over the whole flat buffer, bit for bit,
    with the same coefficient."""
    plan = o.plan(w.numels, w.tied_to, world=w.world, align=w.align)
    P, P_pad, S, N = plan["P"], plan["P_pad"], plan["S"], w.world
    master0 = synth.fill(P_pad, seed=w.seed, stream=synth.STREAM_MASTER, sigma=w.master_sigma,
                         p_limit=P)
    full_st = [master0.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)]
    full_acc = np.zeros(P_pad, np.float32)
    full_params = np.zeros(P_pad * N, np.uint16)
    sh = [[master0[r * S:(r + 1) * S].copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)]
          for r in range(N)]
    sh_acc = [np.zeros(S, np.float32) for _ in range(N)]
    max_norm = None
    for t in range(1, steps + 1):
        for k in range(G):
            local = [synth.fill(P_pad, seed=w.seed, rank=j, step=2000 * t + k,
                                sigma=w.grad_sigma, p_limit=P, bf16=True) for j in range(N)]
            slices = [[local[j][r * S:(r + 1) * S].copy() for j in range(N)] for r in range(N)]
            if k < G - 1:
                o.grad_accumulate(world=N, S=P_pad, lo=0, hi=P_pad, grads=local, accum=full_acc,
                                  first=k == 0)
                for r in range(N):
                    o.grad_accumulate(world=N, S=S, lo=0, hi=S, grads=slices[r], accum=sh_acc[r],
                                      first=k == 0)
                continue
            sq_full = o.grad_sqnorm_accumulated(world=N, S=P_pad, lo=0, hi=P_pad, grads=local,
                                                accum=full_acc, micro_steps=G)
            if max_norm is None:
                max_norm = 0.5 * float(np.sqrt(sq_full))
            c_full, bad_full = o.clip_coef([sq_full], max_norm)
            o.shard_step_accumulated_clipped(world=N, rank=0, S=P_pad, lo=0, hi=P_pad,
                                             grads=local, accum=full_acc, micro_steps=G,
                                             master=full_st[0], m=full_st[1], v=full_st[2],
                                             full_flat=full_params, coef=c_full, skip=bad_full,
                                             t=t, **HP)
            partial = [o.grad_sqnorm_accumulated(world=N, S=S, lo=0, hi=S, grads=slices[r],
                                                 accum=sh_acc[r], micro_steps=G)
                       for r in range(N)]
            c_sh, bad_sh = o.clip_coef(partial, max_norm)
            assert bad_sh == bad_full == 0 and c_sh == c_full and c_sh < 1, (c_sh, c_full)
            fulls = []
            for r in range(N):
                f = np.zeros(P_pad, np.uint16)
                o.shard_step_accumulated_clipped(world=N, rank=r, S=S, lo=0, hi=S,
                                                 grads=slices[r], accum=sh_acc[r],
                                                 micro_steps=G, master=sh[r][0], m=sh[r][1],
                                                 v=sh[r][2], full_flat=f, coef=c_sh,
                                                 skip=bad_sh, t=t, **HP)
                fulls.append(f[r * S:(r + 1) * S].copy())
            gathered = np.zeros(P_pad, np.uint16)
            o.gather(world=N, S=S, elem_size=2, shards=fulls, full_flat=gathered)
            assert np.array_equal(gathered, full_params[:P_pad]), f"params differ at t={t}"
            for i in range(3):
                assert np.array_equal(np.concatenate([x[i] for x in sh]).view(np.uint32),
                                      full_st[i].view(np.uint32)), f"state {i} differs at t={t}"


# ------------------------------------------- per-parameter row sharding ----
def _rows_case_bits(rng, rp, numels, elem):
    """Random bit patterns for each owner parameter (uint8 views)."""
    out = []
    for i, n in enumerate(numels):
        tied = rp["tied"] is not None and rp["tied"][i] >= 0
        out.append(None if tied else rng.integers(0, 256, size=n * elem, dtype=np.uint8))
    return out


def pin_rows_bruteforce(o):
    """All lists of up to 2 parameters (dim0 0..5, 1..3 elements per row, with
    and without a tie), N in 1..5, align in {1, 4}: c = ceil(dim0/N), the N
    chunks tile the rows exactly once (empty chunks for high ranks), S is the
    least multiple of align holding the chunks, and shard -> gather -> unshard
    is the identity on random bits with zero padding."""
    rng = np.random.default_rng(5)
    shapes = [(d, w) for d in range(0, 6) for w in range(1, 4)]
    for k in (1, 2):
        for combo in itertools.product(shapes, repeat=k):
            ties_opts = [None]
            if k == 2 and combo[0] == combo[1]:
                ties_opts.append([-1, 0])
            for ties in ties_opts:
                dim0 = [d for d, _ in combo]
                numels = [d * w for d, w in combo]
                for world in range(1, 6):
                    for align in (1, 4):
                        _check_rows_case(o, rng, dim0, numels, ties, world, align)


def _check_rows_case(o, rng, dim0, numels, ties, world, align, elem=2):
    rp = o.rows_plan(dim0, numels, ties, world=world, align=align)
    used = 0
    for i, (d, n) in enumerate(zip(dim0, numels)):
        if ties is not None and ties[i] >= 0:
            assert rp["offsets"][i] == rp["offsets"][ties[i]]
            continue
        c = rp["rows_per_rank"][i]
        assert c == -(-d // world)
        covered = []
        for r in range(world):
            lo, hi = r * c, min((r + 1) * c, d)
            covered += list(range(lo, max(lo, hi)))
        assert covered == list(range(d))
        assert rp["offsets"][i] == used
        used += c * (n // d if d else 0)
    assert rp["S"] % align == 0 and used <= rp["S"] < used + align
    S = rp["S"]
    params = _rows_case_bits(rng, rp, numels, elem)
    locals_ = []
    for r in range(world):
        loc = np.full(S * elem, 0xEE, np.uint8)
        o.shard_rows(rp, r, elem, params, loc)
        locals_.append(loc)
    gathered = np.concatenate(locals_) if locals_ else np.zeros(0, np.uint8)
    outs = [None if p is None else np.full(p.size, 0xCD, np.uint8) for p in params]
    o.unshard(rp, gathered, elem, outs)
    for p, q in zip(params, outs):
        if p is not None:
            assert np.array_equal(p, q)
    # padding rows and the tail are zero
    for r, loc in enumerate(locals_):
        mask = np.zeros(S * elem, bool)
        for i, (d, n) in enumerate(zip(dim0, numels)):
            if params[i] is None or d == 0:
                continue
            w = n // d
            c = rp["rows_per_rank"][i]
            rows = max(0, min((r + 1) * c, d) - r * c)
            a = rp["offsets"][i] * elem
            mask[a:a + rows * w * elem] = True
        assert not loc[~mask].any(), "padding is not zero"


def pin_rows_pages_layernorm(o):
    """[Dissection] §7: a 768-element layer norm sharded over 64 ranks gives
    12-element shards."""
    g = read_golden_ledger()
    rp = o.rows_plan([768], [768], world=64, align=1)
    assert rp["rows_per_rank"][0] * rp["row_elems"][0] == g["layernorm_768_dp64_shard"][0]


def pin_rows_reshard(o):
    """Resharding to a smaller world M (an integer reshard_after_forward): the
    M-way chunks are the full rows [r*ceil(d/M), ...), and gathering them back
    over M ranks restores the parameters."""
    rng = np.random.default_rng(6)
    dim0, numels = [2048, 256, 11008, 7, 1], [2048, 256 * 2048, 11008 * 4, 7 * 3, 5]
    elem = 2
    full = [rng.integers(0, 256, size=n * elem, dtype=np.uint8) for n in numels]
    for N, M in ((8, 4), (8, 2), (64, 8), (5, 3)):
        rpN = o.rows_plan(dim0, numels, world=N, align=16)
        rpM = o.rows_plan(dim0, numels, world=M, align=16)
        locN = [np.zeros(rpN["S"] * elem, np.uint8) for _ in range(N)]
        for r in range(N):
            o.shard_rows(rpN, r, elem, full, locN[r])
        back = [np.zeros(n * elem, np.uint8) for n in numels]
        o.unshard(rpN, np.concatenate(locN), elem, back)
        for r in range(M):
            loc = np.zeros(rpM["S"] * elem, np.uint8)
            o.shard_rows(rpM, r, elem, back, loc)
            for i, (d, n) in enumerate(zip(dim0, numels)):
                w, c = n // d, -(-d // M)
                rows = max(0, min((r + 1) * c, d) - r * c)
                a = rpM["offsets"][i] * elem
                expect = full[i][r * c * w * elem:(r * c + rows) * w * elem]
                assert np.array_equal(loc[a:a + rows * w * elem], expect), (N, M, r, i)


def pin_rows_ddp_equivalence(o, steps=2):
    """The sharded step on the row layout (each rank's slices are its chunks of
    the N source ranks' gradients), gathered and copied out, equals the
    unsharded DDP step on every parameter, bit for bit; so do master, m, v."""
    dim0 = [1000, 96, 96, 3, 50]
    numels = [1000 * 64, 96 * 64, 96 * 64, 3 * 64, 50]
    ties = [-1, -1, 1, -1, -1]
    N = 4
    rp = o.rows_plan(dim0, numels, ties, world=N, align=128)
    S = rp["S"]
    owners = [i for i in range(len(numels)) if ties[i] < 0]
    fp = o.plan([numels[i] for i in owners], None, world=1, align=1)   # DDP: one flat buffer
    P = fp["P"]
    master_full = synth.fill(P, seed=3, stream=synth.STREAM_MASTER, sigma=0.02)
    ddp = dict(master=master_full.copy(), m=np.zeros(P, np.float32), v=np.zeros(P, np.float32),
               params=np.zeros(P, np.uint16))

    def split(flat):
        return [flat[fp["offsets"][k]:fp["offsets"][k] + numels[i]]
                for k, i in enumerate(owners)]

    def per_param(parts):
        out, k = [], 0
        for i in range(len(numels)):
            if ties[i] >= 0:
                out.append(None)
            else:
                out.append(np.ascontiguousarray(parts[k]))
                k += 1
        return out

    state = []
    for r in range(N):
        st = []
        for arr in (ddp["master"], ddp["m"], ddp["v"]):
            loc = np.zeros(S * 4, np.uint8)
            o.shard_rows(rp, r, 4, [None if x is None else x.view(np.uint8)
                                    for x in per_param(split(arr))], loc)
            st.append(loc.view(np.float32))
        state.append(st)
    for t in range(1, steps + 1):
        local = [synth.fill(P, seed=3, rank=j, step=t, bf16=True) for j in range(N)]
        o.ddp_step(world=N, P_pad=P, local_grads=local, **ddp, t=t, **HP)
        fulls = []
        for r in range(N):
            slices = []
            for j in range(N):
                loc = np.zeros(S * 2, np.uint8)
                o.shard_rows(rp, r, 2, [None if x is None else x.view(np.uint8)
                                        for x in per_param(split(local[j]))], loc)
                slices.append(loc.view(np.uint16))
            f = np.zeros(S * N, np.uint16)
            o.shard_step(world=N, rank=r, S=S, lo=0, hi=S, grads=slices, master=state[r][0],
                         m=state[r][1], v=state[r][2], full_flat=f, t=t, **HP)
            fulls.append(f[r * S:(r + 1) * S].copy())
        gathered = np.concatenate(fulls)
        outs = [None if ties[i] >= 0 else np.zeros(numels[i], np.uint16) for i in range(len(numels))]
        o.unshard(rp, gathered.view(np.uint8), 2, [None if x is None else x.view(np.uint8) for x in outs])
        for k, i in enumerate(owners):
            assert np.array_equal(outs[i], split(ddp["params"])[k]), f"param {i} at t={t}"
        for idx, name in enumerate(("master", "m", "v")):
            g = np.concatenate([state[r][idx] for r in range(N)])
            back = [None if ties[i] >= 0 else np.zeros(numels[i], np.float32) for i in range(len(numels))]
            o.unshard(rp, g.view(np.uint8), 4, [None if x is None else x.view(np.uint8) for x in back])
            for k, i in enumerate(owners):
                assert np.array_equal(back[i].view(np.uint32),
                                      split(ddp[name])[k].view(np.uint32)), f"{name} {i} t={t}"


# ------------------------------------------------ sharded checkpoint ----
def _codes(numels, ties, start=1):
    """Distinct float32 codes per element of every owner parameter."""
    out, c = [], start
    for n, t in zip(numels, ties):
        if t >= 0:
            out.append(None)
            continue
        out.append(np.arange(c, c + n, dtype=np.float32))
        c += n
    return out


def pin_reshard_hand_examples(o):
    """Restores worked by hand from the definition (each shard a piece of the
    global tensors, cut again for the new world or layout):
    flat [5, 3] over 2 ranks -> 3 ranks; FSDP2 rows (A: 3 rows x 2, B: 1 row
    x 4) over 2 ranks -> flat over 1 and over 4 ranks; a tied list."""
    flat2 = ("flat", [5, 3], None, 2, 1)
    old = [np.array([1, 2, 3, 4], np.float32), np.array([5, 6, 7, 8], np.float32)]
    assert o.global_params(flat2, old)[1].tolist() == [6, 7, 8]
    want3 = [[1, 2, 3], [4, 5, 6], [7, 8, 0]]
    for r in range(3):
        assert o.reshard(flat2, old, ("flat", [5, 3], None, 3, 1), r).tolist() == want3[r]
    rp = o.rows_plan([3, 1], [6, 4], None, world=2, align=1)
    assert rp["S"] == 8
    A, B = np.arange(1, 7, dtype=np.float32), np.arange(7, 11, dtype=np.float32)
    rows = ("rows", rp)
    old = [o.shard_of(rows, [A, B], r) for r in range(2)]
    assert old[0].tolist() == [1, 2, 3, 4, 7, 8, 9, 10]
    assert old[1].tolist() == [5, 6, 0, 0, 0, 0, 0, 0]
    assert o.reshard(rows, old, ("flat", [6, 4], None, 1, 1), 0).tolist() == list(range(1, 11))
    want4 = [[1, 2, 3], [4, 5, 6], [7, 8, 9], [10, 0, 0]]
    for r in range(4):
        assert o.reshard(rows, old, ("flat", [6, 4], None, 4, 1), r).tolist() == want4[r]
    tied = ("flat", [4, 2, 4], [-1, -1, 0], 2, 1)
    old = [np.array([1, 2, 3], np.float32), np.array([4, 5, 6], np.float32)]
    got = o.global_params(tied, old)
    assert got[0].tolist() == [1, 2, 3, 4] and got[1].tolist() == [5, 6] and got[2] is None
    assert o.reshard(tied, old, ("flat", [4, 2, 4], [-1, -1, 0], 1, 1), 0).tolist() == \
        [1, 2, 3, 4, 5, 6]


def _random_layouts(o, rng, dims, numels, ties):
    out = []
    for _ in range(3):
        world = int(rng.choice([1, 2, 3, 4, 8, 16]))
        align = int(rng.choice([1, 4, 128]))
        if rng.random() < 0.5:
            out.append(("flat", numels, ties, world, align))
        else:
            out.append(("rows", o.rows_plan(dims, numels, ties, world=world, align=align)))
    return out


def _world(layout):
    return layout[3] if layout[0] == "flat" else layout[1]["world"]


def pin_reshard_invariants(o):
    """For random parameter lists and layouts: a restore into the same layout
    returns every shard unchanged; old -> new -> old is the identity; across
    the new ranks every element code appears exactly once and everything
    else is padding (0)."""
    rng = np.random.default_rng(41)
    for case in range(25):
        k = int(rng.integers(1, 7))
        dims, numels, ties = [], [], []
        for i in range(k):
            if i > 0 and rng.random() < 0.2:
                j = int(rng.integers(0, i))
                while ties[j] >= 0:
                    j = ties[j]
                dims.append(dims[j]); numels.append(numels[j]); ties.append(j)
                continue
            d = int(rng.integers(0, 40))
            dims.append(d); numels.append(d * int(rng.integers(1, 9))); ties.append(-1)
        codes = _codes(numels, ties)
        total = sum(len(c) for c in codes if c is not None)
        a, b, _ = _random_layouts(o, rng, dims, numels, ties)
        A = [o.shard_of(a, codes, r) for r in range(_world(a))]
        for r in range(_world(a)):
            assert np.array_equal(o.reshard(a, A, a, r), A[r]), (case, "identity")
        Bs = [o.reshard(a, A, b, r) for r in range(_world(b))]
        back = [o.reshard(b, Bs, a, r) for r in range(_world(a))]
        for r in range(_world(a)):
            assert np.array_equal(back[r], A[r]), (case, "round trip")
        allv = np.concatenate(Bs)
        nz = np.sort(allv[allv != 0])
        assert np.array_equal(nz, np.arange(1, total + 1, dtype=np.float32)), case


def pin_reshard_next_update(o, steps=3):
    """The pages' test of a restore: the next update after it equals that of
    the uninterrupted run. N = 4 ranks take three steps; the state is
    restored into M = 2 ranks (and into the row layout over 8); step 4 with
    every rank's gradient equal to the same bf16 x (so the mean is exactly x
    at any power-of-two world) gives the uninterrupted run's global master,
    m, v and parameters, bit for bit."""
    w = TINY
    numels, ties = w.numels, w.tied_to
    N = 4
    fl = ("flat", numels, ties, N, w.align)
    pl = o.plan(numels, ties, world=N, align=w.align)
    S, P = pl["S"], pl["P"]
    st = [[synth.fill(S, index0=r * S, seed=2, stream=synth.STREAM_MASTER, sigma=0.02,
                      p_limit=P), np.zeros(S, np.float32), np.zeros(S, np.float32)]
          for r in range(N)]

    def step(state, t, grads_of_rank, world):
        Sx = state[0][0].size
        fulls = []
        for r in range(world):
            f = np.zeros(Sx * world, np.uint16)
            o.shard_step(world=world, rank=r, S=Sx, lo=0, hi=Sx, grads=grads_of_rank(r),
                         master=state[r][0], m=state[r][1], v=state[r][2], full_flat=f, t=t,
                         **HP)
            fulls.append(f[r * Sx:(r + 1) * Sx])
        return fulls

    for t in range(1, steps + 1):
        step(st, t, lambda r: [synth.fill(S, index0=r * S, seed=2, rank=j, step=t,
                                              p_limit=P, bf16=True) for j in range(N)], N)
    x_full = synth.fill(pl["P_pad"], seed=9, step=99, p_limit=P, bf16=True)
    cont = [[a.copy() for a in s] for s in st]
    step(cont, steps + 1, lambda r: [x_full[r * S:(r + 1) * S]] * N, N)
    want = [o.global_params(fl, [cont[r][k] for r in range(N)]) for k in range(3)]
    # x per parameter as fp32 (bf16 bits widened), to cut for the new layouts
    x32 = (x_full.astype(np.uint32) << 16).view(np.float32)
    x_params = o.global_params(fl, [x32[r * S:(r + 1) * S] for r in range(N)])
    dims = [p.shape[0] for p in w.params]
    for new in (("flat", numels, ties, 2, w.align),
                ("rows", o.rows_plan(dims, numels, ties, world=8, align=w.align))):
        M = _world(new)
        rs = [[o.reshard(fl, [st[r][k] for r in range(N)], new, q) for k in range(3)]
              for q in range(M)]
        xq = [o.shard_of(new, x_params, q) for q in range(M)]
        bits = [o.bf16(x) for x in xq]   # x is bf16-exact: the cast gives it back
        step(rs, steps + 1, lambda q: [bits[q]] * M, M)
        for k, name in enumerate(("master", "m", "v")):
            got = o.global_params(new, [rs[q][k] for q in range(M)])
            for i, (g, e) in enumerate(zip(got, want[k])):
                if e is not None:
                    assert np.array_equal(g.view(np.uint32), e.view(np.uint32)), (new[0], name, i)


ALL_PINS = [
    pin_cast_ranges,
    pin_sign_law, pin_zero_grad, pin_constant_grad, pin_eps_placement, pin_lr0_wd0,
    pin_fp64_bound, pin_bias_correction_t2, pin_reduce_dyadic, pin_reduce_order,
    pin_reduce_mean, pin_cast_sampled, pin_param_store, pin_plan_bruteforce,
    pin_plan_buckets, pin_plan_workloads, pin_ledger_pages, pin_ddp_equivalence,
    pin_bucket_invariance, pin_sqnorm_dyadic, pin_clip_coef_closed_forms,
    pin_clip_unit_identity, pin_clip_post_norm, pin_clip_skip, pin_clip_ddp_equivalence,
    pin_accum_single_microstep_identity, pin_accum_dyadic, pin_accum_equals_merged,
    pin_accum_first_overwrites, pin_accum_ddp_equivalence, pin_accum_clip_reductions,
    pin_accum_clip_dyadic, pin_accum_clip_ddp_equivalence, pin_rows_bruteforce,
    pin_rows_pages_layernorm, pin_rows_reshard, pin_rows_ddp_equivalence,
    pin_reshard_hand_examples, pin_reshard_invariants, pin_reshard_next_update,
    pin_ddp_equivalence_gpt2_buckets,
]
