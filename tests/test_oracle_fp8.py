"""Pins of the FP8 (E4M3) part of the oracle: the codec against the format's published
constants, exhaustive round trips, ties-to-even at every midpoint and torch's own E4M3
conversion; the FP8 attention oracle (numpy) against the bf16 C oracle on the same values
(every E4M3 value is a bf16 value, and power-of-two scales keep them exact)."""
import numpy as np
import pytest

import oracle
import synth


def test_published_constants():
    enc = lambda v: int(oracle.e4m3_encode([v])[0])
    assert enc(448.0) == 0x7E and oracle.e4m3_decode([0x7E])[0] == 448.0          # largest finite
    assert enc(2.0 ** -6) == 0x08 and oracle.e4m3_decode([0x08])[0] == 2.0 ** -6  # smallest normal
    assert enc(2.0 ** -9) == 0x01 and oracle.e4m3_decode([0x01])[0] == 2.0 ** -9  # smallest subnormal
    assert enc(1.0) == 0x38 and enc(-2.0) == 0xC0
    assert np.isnan(oracle.e4m3_decode([0x7F, 0xFF])).all()                        # S.1111.111: NaN
    assert enc(1e30) == 0x7E and enc(-1e30) == 0xFE and enc(np.inf) == 0x7E         # saturating
    assert enc(float("nan")) == 0x7F


def test_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_midpoints_round_to_even():
    pos = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    got = oracle.e4m3_encode(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    # just off the midpoints, the nearer code wins
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mids, -np.inf)), lo.astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mids, np.inf)), (lo + 1).astype(np.uint8))


def test_agrees_with_torch_conversion():
    torch = pytest.importorskip("torch")
    x = np.concatenate([np.random.default_rng(3).normal(0, s, 20000) for s in (0.01, 1, 100)])
    x = np.clip(x, -448, 448).astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x.astype(np.float64)), t)


def _fp8_workload(seed, lens, hq, hkv, d, p, window=0):
    """A GQA workload whose K/V are E4M3 codes (drawn values encoded by the oracle)."""
    w = synth.make_gqa(seed, lens, hq, hkv, d, p, window=window)
    kc = oracle.e4m3_encode(synth.bf16_bits_to_f32(w.k_pool).astype(np.float64) * 4.0)
    vc = oracle.e4m3_encode(synth.bf16_bits_to_f32(w.v_pool).astype(np.float64) * 4.0)
    return w, kc, vc


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 8.0)])
def test_fp8_attention_equals_bf16_oracle_on_the_same_values(k_scale, v_scale):
    w, kc, vc = _fp8_workload(61, [1, 31, 33, 100, 0], 8, 2, 64, 16, window=40)
    o, l = oracle.gqa_fp8(w.q, kc, vc, w.layout.block_table, w.layout.context_lens, w.scale, k_scale, v_scale,
                          w.window)
    # the same values as bf16 bit patterns (exact: E4M3 values times powers of two are bf16 values)
    kb = synth.f32_to_bf16_bits((oracle.e4m3_decode(kc) * k_scale).astype(np.float32))
    vb = synth.f32_to_bf16_bits((oracle.e4m3_decode(vc) * v_scale).astype(np.float32))
    ro, rl = oracle.gqa(w.q, kb, vb, w.layout.block_table, w.layout.context_lens, w.scale, w.window)
    assert np.abs(o - ro).max() < 1e-12
    both = np.isinf(l) & np.isinf(rl)
    with np.errstate(invalid="ignore"):
        assert np.all(np.where(both, 0.0, np.abs(l - rl)) < 1e-12)


def test_fp8_write_round_trip():
    w = synth.make_kv_write(62, 40, 2, 64, 8, 8)
    # rows that are exactly E4M3 values times the scale survive the write unchanged
    codes = np.random.default_rng(5).integers(0, 126, size=w.k.shape).astype(np.uint8)
    vals = (oracle.e4m3_decode(codes) * 0.5).astype(np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    kp, _ = oracle.kv_write_fp8(bits, bits, w.slots, np.zeros(w.pool_shape(), np.uint8),
                                np.zeros(w.pool_shape(), np.uint8), 0.5, 0.5)
    P = w.page_size
    assert np.array_equal(kp[w.slots // P, w.slots % P], codes)
