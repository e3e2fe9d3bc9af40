"""The seeded generator: published splitmix64 values, bf16 rounding, layout invariants."""
import numpy as np
import torch

import synth


def test_splitmix64_published_values():
    # splitmix64 seeded with 0: first outputs as published with the reference C implementation
    out = synth.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [hex(int(x)) for x in out] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4", "0x6c45d188009454f"]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -1e-40], dtype=np.float32)])
    ours = synth.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(synth.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_normal_moments():
    z = synth.normal(123, np.arange(200000, dtype=np.uint64))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def test_permutation_is_a_permutation():
    p = synth.permutation(5, 1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not np.array_equal(p, np.arange(1000))


def test_layout_and_poison():
    w = synth.make_gqa(3, [1, 31, 32, 33, 100], 4, 2, 64, 32, window=40)
    bt = w.layout.block_table
    used = [int(p) for p in bt.ravel() if p >= 0]
    assert len(used) == len(set(used)) == w.layout.num_pages
    # row 4 (L=100, window 40): tokens [60, 100) visible; page 0 (tokens 0..31) never read -> NaN
    nan = synth.BF16_NAN
    assert (w.k_pool[bt[4, 0]] == nan).all()
    assert (w.k_pool[bt[4, 1], : 60 - 32] == nan).all() and not (w.k_pool[bt[4, 1], 60 - 32:] == nan).any()
    assert (w.v_pool[bt[4, 3], 100 - 96:] == nan).all()
    # row 0 (L=1): slot 0 data, the rest poisoned
    assert not (w.k_pool[bt[0, 0], 0] == nan).any() and (w.k_pool[bt[0, 0], 1:] == nan).all()


def test_same_logical_data_under_any_page_order():
    a = synth.make_gqa(9, [40, 70], 2, 1, 32, 16, scramble=True)
    b = synth.make_gqa(9, [40, 70], 2, 1, 32, 16, scramble=False)
    for r, L in enumerate([40, 70]):
        for lp in range((L + 15) // 16):
            assert np.array_equal(a.k_pool[a.layout.block_table[r, lp]], b.k_pool[b.layout.block_table[r, lp]])


def test_workload_shapes():
    w = synth.workload("tiny")
    assert w.q.shape == (6, 8, 128) and w.k_pool.shape[1:] == (32, 2, 128)
    assert list(w.layout.context_lens) == [1, 31, 32, 33, 64, 100]
    lens = synth.context_lengths(20263, 16, "uniform", 2048, 32768)
    assert lens.min() >= 2048 and lens.max() <= 32768
    lens = synth.context_lengths(20262, 32, "loguniform", 128, 16384)
    assert lens.min() >= 128 and lens.max() <= 16384


def test_fp8_codes_recipe():
    """FP8 pools: visible slots hold finite E4M3 codes (never S.1111.111), drawn per the recipe
    (about 1/32 from all 127 magnitudes, the rest from 0x28..0x6F), and every slot no row may
    read holds the NaN code 0x7F; the same logical codes under any page order."""
    codes = synth.e4m3_codes(synth.stream_seed(5, synth.TAG_K), np.arange(200000, dtype=np.uint64))
    mag = codes & 0x7F
    assert not np.any(mag == 0x7F)
    wide = (mag < 0x28) | (mag > 0x6F)
    assert 0.01 < wide.mean() < 0.03                      # the 1/32 arm, outside the narrow range
    assert {0x00, 0x01, 0x7E} <= set(np.unique(mag).tolist())  # zero, smallest subnormal, 448
    assert 0.45 < (codes >> 7).mean() < 0.55               # signs balanced
    w = synth.make_gqa(9, [1, 31, 40], 8, 2, 128, 16, fp8=True, window=20)
    wi = synth.make_gqa(9, [1, 31, 40], 8, 2, 128, 16, fp8=True, window=20, scramble=False)
    bt, P = w.layout.block_table, w.layout.page_size
    seen = np.zeros(w.k_pool.shape[:2], dtype=bool)
    for b, L in enumerate(w.layout.context_lens):
        lo, hi = synth.visible_range(int(L), w.window)
        t = np.arange(lo, hi)
        pk = w.k_pool[bt[b, t // P], t % P]
        assert not np.any((pk & 0x7F) == 0x7F)
        assert np.array_equal(pk, wi.k_pool[wi.layout.block_table[b, t // P], t % P])
        seen[bt[b, t // P], t % P] = True
    assert np.all(w.k_pool[~seen] == synth.E4M3_NAN) and np.all(w.v_pool[~seen] == synth.E4M3_NAN)


def test_nvfp4_rows_recipe():
    """NVFP4 pools: visible rows hold uniform code bytes, block-scale codes drawn per the recipe
    (about 1/32 from 0x00..0x4F, the rest from 0x28..0x47, never NaN) and zero padding; every
    slot no row may read holds 0x7F in every byte; the same logical rows under any page order."""
    D = 128
    R = synth.nvfp4_row_bytes(D)
    assert R == 80 and synth.nvfp4_row_bytes(64) == 48 and synth.nvfp4_row_bytes(256) == 144
    b = synth.nvfp4_bytes(synth.stream_seed(5, synth.TAG_K), np.arange(R * 4000, dtype=np.uint64), D)
    rows = b.reshape(4000, R)
    codes, scales, pad = rows[:, : D // 2], rows[:, D // 2: D // 2 + D // 16], rows[:, D // 2 + D // 16:]
    assert not pad.any()
    assert len(np.unique(codes)) == 256                     # every code byte occurs
    assert scales.max() <= 0x4F and not np.any(scales == 0x7F)
    wide = (scales < 0x28) | (scales > 0x47)
    assert 0.005 < wide.mean() < 0.04
    assert {0x00, 0x01} <= set(np.unique(scales).tolist())  # zero and the smallest subnormal scale
    w = synth.make_gqa(9, [1, 31, 40], 8, 2, D, 16, nvfp4=True, window=20)
    wi = synth.make_gqa(9, [1, 31, 40], 8, 2, D, 16, nvfp4=True, window=20, scramble=False)
    assert w.k_pool.shape[2:] == (2, R) and w.k_pool.dtype == np.uint8
    bt, P = w.layout.block_table, w.layout.page_size
    seen = np.zeros(w.k_pool.shape[:2], dtype=bool)
    for bi, L in enumerate(w.layout.context_lens):
        lo, hi = synth.visible_range(int(L), w.window)
        t = np.arange(lo, hi)
        pk = w.k_pool[bt[bi, t // P], t % P]
        assert not pk[..., D // 2 + D // 16:].any()
        assert np.array_equal(pk, wi.k_pool[wi.layout.block_table[bi, t // P], t % P])
        seen[bt[bi, t // P], t % P] = True
    assert np.all(w.k_pool[~seen] == 0x7F) and np.all(w.v_pool[~seen] == 0x7F)
    # the algorithmic bytes count 9/16 byte per cached value
    vis = w.visible_tokens()
    assert w.algorithmic_bytes() == vis * 2 * 2 * (D * 9 // 16) + 3 * 8 * D * 2 + 3 * 8 * (D * 2 + 4)
