"""The division-free Q8_0 code used by the CUDA quantizers, checked on the CPU.

The kernels never divide x by d for the activation code.  They form
y = x * r with r an approximate reciprocal of d (within one ulp) and take the
nearest integer of y; only when y lies within 2^-14 of a half-integer do they
decide the rounding of the IEEE quotient exactly, from the sign of |x| - m d
(m the midpoint below the half-integer h), computed as two fused
multiply-adds.  A scale below 2^-60 is first multiplied, with x, by 2^64.

This test restates that procedure in numpy (f32 steps in f32; the fused
multiply-adds exactly in f64, which is what a single rounding of an exact
value keeps: its sign and its zero) and compares it with the definition,
roundf(x / d) clamped to [-127, 127] with the IEEE f32 quotient, on values
placed on and beside the rounding ties, on random blocks and on subnormal
scales.  The GPU tests compare the kernels' codes with the oracle on the same
kinds of inputs; this one pins the reasoning the kernels rely on, for many
more values than a GPU test reads back.
"""
import numpy as np

F32 = np.float32


def q8_reference(x, d):
    """roundf(x / d) with the IEEE f32 quotient, clamped; 0 when d = 0."""
    with np.errstate(all="ignore"):
        q = np.where(d == 0, F32(0), x / np.where(d == 0, F32(1), d)).astype(F32)
    c = np.trunc(q.astype(np.float64) + np.copysign(0.5, q))
    return np.clip(c, -127, 127).astype(np.int64)


def q8_division_free(x, d, rng):
    s = np.where(d < F32(2.0 ** -60), F32(2.0 ** 64), F32(1)).astype(F32)
    ds = (d * s).astype(F32)
    with np.errstate(all="ignore"):
        r = (F32(1) / np.where(ds == 0, F32(1), ds)).astype(F32)
    # rcp.approx.f32 is within one ulp: move r by up to one ulp either way
    step = rng.integers(0, 3, r.size)
    r = np.where(step == 1, np.nextafter(r, F32(np.inf)), np.where(step == 2, np.nextafter(r, F32(0)), r)).astype(F32)
    r = np.where(d == 0, F32(0), r)
    xs = (x * s).astype(F32)
    y = (xs * r).astype(F32)
    n = np.rint(y).astype(F32)
    away = np.abs((y - n).astype(F32)) < F32(0.5) - F32(2.0 ** -14)
    k = np.floor(np.abs(y)).astype(F32)
    h = (k + F32(0.5)).astype(F32)
    u = (h - (h.view(np.int32) - 1).view(F32)).astype(F32)
    e = np.abs(xs).astype(np.float64) - h.astype(np.float64) * ds.astype(np.float64)
    # e is exact in f32 wherever the near-tie branch is used
    assert np.all(away | (e.astype(F32).astype(np.float64) == e))
    t = (F32(0.5) * u).astype(np.float64) * ds.astype(np.float64) + e
    up = (t > 0) | ((t == 0) & ((h.view(np.int32) & 1) == 0))
    c = k.astype(np.int64) + up
    c = np.where(xs < 0, -c, c)
    c = np.where(away, n.astype(np.int64), c)
    return np.clip(c, -127, 127)


def blocks_near_ties(rng, n, kind):
    if kind == 0:
        amax = np.exp(rng.uniform(-103, 80, n)).astype(F32)        # down to subnormal scales
    elif kind == 1:
        amax = (rng.uniform(0, 1, n) * 2.0 ** -120).astype(F32)   # subnormal scales only
    else:
        amax = np.exp(rng.uniform(-20, 20, n)).astype(F32)
    d = (amax / F32(127)).astype(F32)
    if kind < 3:
        k = rng.integers(0, 128, n).astype(np.float64)
        x = ((k + 0.5) * d.astype(np.float64)).astype(F32)
        for _ in range(rng.integers(0, 3)):
            st = rng.integers(-1, 2, n)
            x = np.where(st > 0, np.nextafter(x, F32(np.inf)),
                         np.where(st < 0, np.nextafter(x, F32(-np.inf)), x)).astype(F32)
    else:
        x = (rng.uniform(-1, 1, n) * amax).astype(F32)
    x = (x * rng.choice([-1, 1], n)).astype(F32)
    return np.clip(x, -amax, amax).astype(F32), d


def test_division_free_code_equals_ieee_quotient():
    rng = np.random.default_rng(20)
    for it in range(64):
        x, d = blocks_near_ties(rng, 1 << 16, it % 4)
        want, got = q8_reference(x, d), q8_division_free(x, d, rng)
        bad = want != got
        assert not bad.any(), f"x={x[bad][0]!r} d={d[bad][0]!r}: {want[bad][0]} vs {got[bad][0]}"


def test_division_free_exact_ties_power_of_two_scales():
    rng = np.random.default_rng(21)
    k = np.arange(-128, 128).astype(np.float64)
    for e in range(-149, 120):
        d = np.full(k.size, F32(2.0 ** e))
        x = ((k + 0.5) * d.astype(np.float64)).astype(F32)
        ok = np.isfinite(x) & (np.abs(x.astype(np.float64)) <= 127.5 * d.astype(np.float64))
        assert np.array_equal(q8_reference(x[ok], d[ok]), q8_division_free(x[ok], d[ok], rng))


def test_zero_scale():
    rng = np.random.default_rng(22)
    x = np.zeros(32, F32)
    d = np.zeros(32, F32)
    assert np.array_equal(q8_division_free(x, d, rng), np.zeros(32, np.int64))
