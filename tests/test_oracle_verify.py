"""Pins of the multi-query (verify) oracle: dense causal attention in torch
float64 over the regenerated logical K/V (a [Q, L] mask), and its reduction to
the decode oracle (one query position; the last position of Q)."""
import numpy as np
import pytest

import oracle
import refs
import synth


def _close(got_o, got_l, ref_o, ref_l, tol=1e-12):
    assert np.abs(got_o - ref_o).max() <= tol
    both = np.isinf(got_l) & np.isinf(ref_l)
    with np.errstate(invalid="ignore"):
        err = np.where(both, 0.0, np.abs(got_l - ref_l))
    assert np.all(err <= tol)


@pytest.mark.parametrize("lens,hq,hkv,d,p,Q,window", [
    ([1, 2, 3, 40, 70, 0], 8, 2, 64, 16, 3, 0),      # rows shorter than Q: early positions see nothing
    ([10, 35, 70], 8, 2, 64, 16, 4, 9),              # a window shorter than the block
    ([33, 64, 100], 4, 1, 32, 8, 7, 0),
    ([200, 129], 20, 2, 64, 32, 2, 50),
])
def test_verify_oracle_equals_dense_causal(lens, hq, hkv, d, p, Q, window):
    w = synth.make_gqa(90 + Q, lens, hq, hkv, d, p, window=window, num_query=Q)
    o, l = oracle.verify_gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                             w.window)
    ro, rl = refs.dense_verify(w)
    _close(o, l, ro.reshape(-1, d), rl.reshape(-1))


def test_one_position_is_the_decode():
    w = synth.make_gqa(95, [1, 31, 32, 33, 64, 100], 8, 2, 64, 16, window=40)
    a = oracle.gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale, w.window)
    b = oracle.verify_gqa(w.q[:, None], w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens,
                          w.scale, w.window)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_last_position_is_the_decode_of_the_whole_row():
    w = synth.make_gqa(96, [5, 50, 99], 8, 2, 64, 16, num_query=4)
    o, l = oracle.verify_gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale, 0)
    d = oracle.gqa(w.q[:, -1], w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale, 0)
    B, Q, Hq, D = w.q.shape
    assert np.array_equal(o.reshape(B, Q, Hq, D)[:, -1].reshape(-1, D), d[0])
