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
