"""The division the quantizing KV writes use for a scale that is not a power of two (Markstein's
correction: y = RN(1/b), q = RN(a y), r = a - b q by one fma, result RN(q + r y); P. Markstein,
IBM J. Res. Dev. 34(1), 1990) equals the correctly rounded float32 quotient RN(a/b).  Checked
here in exact rational arithmetic on float32 operands of the ranges the writes divide: bf16 values
by pool scales in [2^-100, 2^100], and float32 quotients by E4M3 block scales (2^-9 .. 448)."""
from fractions import Fraction

import numpy as np

import synth


def rn32(x: Fraction) -> np.float32:
    """Round a rational to the nearest float32, ties to even (normal range)."""
    c = np.float32(float(x))  # within one float32 ulp of x
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - x)
        if best is None or d < best[0] or (d == best[0] and (int(cand.view(np.uint32)) & 1) == 0):
            best = (d, cand)
    return best[1]


def fma32(a, b, c) -> np.float32:
    return rn32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def markstein(a: np.float32, b: np.float32) -> np.float32:
    y = rn32(1 / Fraction(float(b)))
    q = np.float32(a * y)          # one float32 product: RN(a y)
    r = fma32(-q, b, a)            # a - b q, rounded once
    return fma32(r, y, q)          # RN(q + r y)


def _check(a_vals, b_vals):
    bad = []
    for a, b in zip(a_vals, b_vals):
        want = rn32(Fraction(float(a)) / Fraction(float(b)))
        got = markstein(a, b)
        if got != want:
            bad.append((float(a), float(b), float(got), float(want)))
    assert not bad, bad[:5]


def test_bf16_values_by_pool_scales():
    rng = np.random.default_rng(5)
    a = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(
        (rng.standard_normal(4000) * np.exp2(rng.integers(-20, 20, 4000))).astype(np.float32)))
    b = (rng.uniform(1, 2, 4000) * np.exp2(rng.integers(-100, 100, 4000))).astype(np.float32)
    keep = np.isfinite(a / b.astype(np.float64)) & (np.abs(a / b.astype(np.float64)) > 2.0 ** -125) & \
        (np.abs(a / b.astype(np.float64)) < 2.0 ** 127)
    _check(a[keep], b[keep])


def test_quotients_by_every_e4m3_block_scale():
    import oracle
    rng = np.random.default_rng(6)
    codes = np.arange(1, 127, dtype=np.uint8)           # every non-zero finite E4M3 value
    ds = oracle.e4m3_decode(codes).astype(np.float32)
    b = np.repeat(ds, 40)
    a = (rng.uniform(-8, 8, b.size) * b).astype(np.float32)   # quotients around the E2M1 range
    _check(a, b)


def test_near_e2m1_midpoints():
    """Dividends placed one ulp around (midpoint x divisor), where a one-ulp error of the quotient
    would flip an E2M1 code."""
    import oracle
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    ds = oracle.e4m3_decode(np.arange(1, 127, dtype=np.uint8)).astype(np.float32)
    a_list, b_list = [], []
    for d in ds:
        for m in mids:
            c = np.float32(m * d)
            for x in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
                a_list.append(x)
                b_list.append(d)
    _check(np.array(a_list, dtype=np.float32), np.array(b_list, dtype=np.float32))
