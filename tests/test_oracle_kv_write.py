"""Pins of the KV-write oracle: the slot convention it writes must be the one the
attention oracle reads (page slot // P, position slot % P), checked against the
generator's own placement of logical tokens; padding and untouched slots stay as
they were."""
import numpy as np

import oracle
import synth


def _slots_of(layout, b, L):
    """Slots of tokens 0..L-1 of row b under the block table (the read convention)."""
    P = layout.page_size
    t = np.arange(L)
    return layout.block_table[b, t // P].astype(np.int64) * P + t % P


def test_write_then_read_matches_generator_placement():
    w = synth.make_gqa(31, [5, 40, 33], 4, 2, 64, 16)
    kp0 = np.full_like(w.k_pool, synth.BF16_NAN)
    vp0 = np.full_like(w.v_pool, synth.BF16_NAN)
    kp, vp = kp0, vp0
    for b, L in enumerate(w.layout.context_lens):
        slots = _slots_of(w.layout, b, int(L))
        P = w.layout.page_size
        # the rows the generator placed for row b, read back at those slots
        k_rows = w.k_pool[slots // P, slots % P]
        v_rows = w.v_pool[slots // P, slots % P]
        kp, vp = oracle.kv_write(k_rows, v_rows, slots, kp, vp)
    assert np.array_equal(kp, w.k_pool) and np.array_equal(vp, w.v_pool)
    # so attention over the written pools is attention over the generator's pools, bit for bit
    a = oracle.gqa(w.q, kp, vp, w.layout.block_table, w.layout.context_lens, w.scale, 0)
    b = oracle.gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_padding_and_untouched_slots():
    w = synth.make_kv_write(7, 50, 2, 64, 8, 12, pad_every=5)
    kp, vp = oracle.kv_write(w.k, w.v, w.slots, w.empty_pool(), w.empty_pool())
    written = np.zeros(w.num_pages * w.page_size, dtype=bool)
    written[w.slots[w.slots >= 0]] = True
    flat_k = kp.reshape(-1, 2, 64)
    assert (flat_k[~written] == synth.BF16_NAN).all()
    for t in range(w.num_tokens):
        s = w.slots[t]
        if s >= 0:
            assert np.array_equal(flat_k[s], w.k[t])
        else:
            assert (t + 1) % 5 == 0


def test_mla_cache_row_is_latent_then_rope():
    w = synth.make_kv_write(9, 20, 0, 0, 16, 4, mla=True)
    cache = oracle.mla_cache_write(w.k, w.v, w.slots, w.empty_pool())
    flat = cache.reshape(-1, 576)
    for t in range(w.num_tokens):
        s = w.slots[t]
        assert np.array_equal(flat[s, :512], w.k[t]) and np.array_equal(flat[s, 512:], w.v[t])


def test_mla_write_then_read_matches_generator_placement():
    w = synth.make_mla(33, [70, 3], 4, 16)
    cache = np.full_like(w.cache, synth.BF16_NAN)
    P = w.layout.page_size
    for b, L in enumerate(w.layout.context_lens):
        slots = _slots_of(w.layout, b, int(L))
        rows = w.cache[slots // P, slots % P]
        cache = oracle.mla_cache_write(rows[:, :512], rows[:, 512:], slots, cache)
    a = oracle.mla(w.q, cache, w.w_uk, w.w_uv, w.layout.block_table, w.layout.context_lens, w.scale)
    b = oracle.mla(w.q, w.cache, w.w_uk, w.w_uv, w.layout.block_table, w.layout.context_lens, w.scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
