"""Pins of the NVFP4 part of the oracle (the quantized KV cache's second format): the E2M1 codec
against the format's definition (magnitudes, exhaustive round trips, ties to even at every
midpoint, saturation), the block quantization against rows built from exact values, the pool
row layout, and the NVFP4 attention oracle (numpy) against the bf16 C oracle on the same values
(every E2M1 value times an E4M3 scale times a power of two is a bf16 value)."""
import numpy as np
import pytest

import oracle
import synth


def test_e2m1_magnitudes_and_signs():
    # the format's eight magnitudes: 0, the subnormal 0.5, then (1 + m / 2) 2^(e - 1)
    assert list(oracle.e2m1_decode(np.arange(8))) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(oracle.e2m1_decode(np.arange(8, 16))) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert np.signbit(oracle.e2m1_decode([8]))[0]


def test_e2m1_round_trip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


def test_e2m1_midpoints_round_to_even_and_saturate():
    mags = oracle.e2m1_decode(np.arange(8))
    mids = (mags[:-1] + mags[1:]) / 2                 # 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
    lo = np.arange(7)
    want = np.where(lo % 2 == 0, lo, lo + 1)          # the code with the even mantissa bit
    assert np.array_equal(oracle.e2m1_encode(mids), want.astype(np.uint8))
    assert np.array_equal(oracle.e2m1_encode(-mids), (want | 8).astype(np.uint8))
    assert np.array_equal(oracle.e2m1_encode(np.nextafter(mids, -np.inf)), lo.astype(np.uint8))
    assert np.array_equal(oracle.e2m1_encode(np.nextafter(mids, np.inf)), (lo + 1).astype(np.uint8))
    assert list(oracle.e2m1_encode([6.0, 6.5, 1e9, np.inf, -np.inf])) == [7, 7, 7, 7, 15]
    assert oracle.e2m1_encode([float("nan")])[0] == 0


def test_block_quantization_of_exact_values():
    """Rows whose 16-value blocks are E2M1 values times an E4M3 value v times the pool scale, each
    block holding a 6 (so its amax / (6 pool_scale) is v exactly): the scale code is v's and every
    value comes back exactly."""
    rng = np.random.default_rng(11)
    pool_scale = 0.25
    n, D = 64, 128
    codes = rng.integers(0, 16, size=(n, D)).astype(np.uint8)
    codes[:, ::16] = rng.choice([7, 15], size=(n, D // 16))        # one +-6 per block
    v_codes = rng.integers(0x08, 0x60, size=(n, D // 16)).astype(np.uint8)  # normal E4M3 scales
    v = oracle.e4m3_decode(v_codes)
    x = (oracle.e2m1_decode(codes).reshape(n, D // 16, 16) * v[..., None] * pool_scale).reshape(n, D)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)   # exact in float32
    got_codes, got_scales = oracle.nvfp4_quantize_rows(x.astype(np.float32), pool_scale)
    assert np.array_equal(got_scales, v_codes)
    # -0 and +0 are both zero: compare the values
    assert np.array_equal(oracle.e2m1_decode(got_codes), oracle.e2m1_decode(codes))
    rows = oracle.nvfp4_pack_rows(got_codes, got_scales)
    assert np.array_equal(oracle.nvfp4_decode_rows(rows, D, pool_scale), x)


def test_block_quantization_rounds_each_value_to_its_nearest_code():
    """Random rows: every decoded value is the nearest E2M1 multiple of its block's decoded scale
    (up to the scale's saturation at 6), and the scale is the nearest E4M3 value of amax / 6."""
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, size=(200, 64)).astype(np.float32)
    codes, scales = oracle.nvfp4_quantize_rows(x, 1.0)
    ds = oracle.e4m3_decode(scales)
    amax = np.abs(x.reshape(200, 4, 16)).max(axis=-1)
    assert np.array_equal(scales, oracle.e4m3_encode((amax.astype(np.float32) / np.float32(6)).astype(np.float64)))
    y = x.reshape(200, 4, 16).astype(np.float64) / ds[..., None]
    grid = oracle.e2m1_decode(np.arange(8))
    got = np.abs(oracle.e2m1_decode(codes).reshape(200, 4, 16))
    best = np.abs(np.abs(y)[..., None] - grid).min(axis=-1)
    assert np.all(np.abs(np.abs(y) - got) <= best + 1e-12)


def test_pool_row_layout():
    D = 64
    codes = np.arange(D, dtype=np.uint8) % 16
    scales = np.array([0x38, 0x40, 0x30, 0x48], dtype=np.uint8)
    row = oracle.nvfp4_pack_rows(codes, scales)
    assert row.shape == (oracle.nvfp4_row_bytes(D),) == (48,)
    assert row[0] == (0 | (1 << 4)) and row[1] == (2 | (3 << 4))      # even dim in the low nibble
    assert list(row[32:36]) == list(scales)                              # then the block scales
    assert not row[36:].any()                                            # then zero padding
    assert oracle.nvfp4_row_bytes(128) == 80 and oracle.nvfp4_row_bytes(256) == 144


def _nvfp4_workload(seed, lens, hq, hkv, d, p, k_scale, v_scale, window=0):
    w = synth.make_gqa(seed, lens, hq, hkv, d, p, window=window)
    kf = synth.bf16_bits_to_f32(w.k_pool)
    vf = synth.bf16_bits_to_f32(w.v_pool)
    kr = oracle.nvfp4_pack_rows(*oracle.nvfp4_quantize_rows(kf, k_scale))
    vr = oracle.nvfp4_pack_rows(*oracle.nvfp4_quantize_rows(vf, v_scale))
    return w, kr, vr


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 2.0)])
def test_nvfp4_attention_equals_bf16_oracle_on_the_same_values(k_scale, v_scale):
    w, kr, vr = _nvfp4_workload(71, [1, 31, 33, 100, 0], 8, 2, 64, 16, k_scale, v_scale, window=40)
    o, l = oracle.gqa_nvfp4(w.q, kr, vr, w.layout.block_table, w.layout.context_lens, w.scale, k_scale, v_scale,
                            w.window)
    D = 64
    kb = synth.f32_to_bf16_bits(oracle.nvfp4_decode_rows(kr, D, k_scale).astype(np.float32))
    vb = synth.f32_to_bf16_bits(oracle.nvfp4_decode_rows(vr, D, v_scale).astype(np.float32))
    # the values are bf16 values: the conversion above is exact
    assert np.array_equal(synth.bf16_bits_to_f32(kb).astype(np.float64), oracle.nvfp4_decode_rows(kr, D, k_scale),
                          equal_nan=True)  # (slots no key uses hold NaN poison)
    ro, rl = oracle.gqa(w.q, kb, vb, w.layout.block_table, w.layout.context_lens, w.scale, w.window)
    assert np.abs(o - ro).max() < 1e-12
    both = np.isinf(l) & np.isinf(rl)
    with np.errstate(invalid="ignore"):
        assert np.all(np.where(both, 0.0, np.abs(l - rl)) < 1e-12)


def test_nvfp4_write_places_rows_at_their_slots():
    w = synth.make_kv_write(72, 40, 2, 64, 8, 8, pad_every=7)
    R = oracle.nvfp4_row_bytes(64)
    pool = np.full((w.num_pages, w.page_size, 2, R), 0xAB, dtype=np.uint8)
    kp, vp = oracle.kv_write_nvfp4(w.k, w.v, w.slots, pool, pool.copy(), 0.5, 1.0)
    kr = oracle.nvfp4_pack_rows(*oracle.nvfp4_quantize_rows(synth.bf16_bits_to_f32(w.k), 0.5))
    P = w.page_size
    for t, s in enumerate(w.slots):
        if s < 0:
            continue
        assert np.array_equal(kp[s // P, s % P], kr[t])
    written = {int(s) for s in w.slots if s >= 0}
    for s in range(w.num_pages * P):
        if s not in written:
            assert (kp[s // P, s % P] == 0xAB).all() and (vp[s // P, s % P] == 0xAB).all()
