"""Paged KV write on the GPU (through the C ABI) against the oracle: bit-exact,
padding skipped, untouched slots unchanged, bad slots reported; and a decode over
pools filled by the GPU write equals the oracle's decode."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def _u16(a):
    return gu.dev(a)


@pytest.mark.parametrize("T,Hkv,D,P,pages,pad", [(1, 1, 64, 8, 1, 0), (37, 2, 128, 16, 8, 5),
                                                  (300, 8, 128, 32, 16, 7), (64, 4, 256, 32, 4, 0),
                                                  (1000, 3, 64, 256, 5, 11)])
def test_kv_write_bit_exact(T, Hkv, D, P, pages, pad):
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(40 + T, T, Hkv, D, P, pages, pad_every=pad)
    kp0, vp0 = w.empty_pool(), w.empty_pool()
    ref_k, ref_v = oracle.kv_write(w.k, w.v, w.slots, kp0, vp0)
    k, v = _u16(w.k), _u16(w.v)
    kp, vp = _u16(kp0), _u16(vp0)
    slots = torch.from_numpy(w.slots).cuda()
    pa.pa_kv_write(k, v, slots, kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(gu.bits(kp), ref_k) and np.array_equal(gu.bits(vp), ref_v)


def test_bad_slot_is_reported_and_skipped():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(50, 20, 2, 64, 8, 4)
    slots = w.slots.copy()
    slots[3] = w.num_pages * w.page_size + 2     # past the pool
    ref_k, ref_v = oracle.kv_write(w.k, w.v, np.where(np.arange(20) == 3, -1, slots), w.empty_pool(),
                                   w.empty_pool())
    kp, vp = _u16(w.empty_pool()), _u16(w.empty_pool())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_kv_write(_u16(w.k), _u16(w.v), torch.from_numpy(slots).cuda(), kp, vp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_SLOT
    assert np.array_equal(gu.bits(kp), ref_k) and np.array_equal(gu.bits(vp), ref_v)


def test_mla_cache_write_bit_exact():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(60, 333, 0, 0, 64, 8, pad_every=9, mla=True)
    ref = oracle.mla_cache_write(w.k, w.v, w.slots, w.empty_pool())
    cache = _u16(w.empty_pool())
    pa.pa_mla_cache_write(_u16(w.k), _u16(w.v), torch.from_numpy(w.slots).cuda(), cache)
    torch.cuda.synchronize()
    assert np.array_equal(gu.bits(cache), ref)


def test_decode_over_gpu_written_pools():
    """Fill empty pools with every visible token through pa_kv_write, then decode."""
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(70, [1, 31, 32, 33, 64, 100, 685, 1000], 16, 2, 128, 32)
    P = w.layout.page_size
    kp = _u16(np.full_like(w.k_pool, synth.BF16_NAN))
    vp = _u16(np.full_like(w.v_pool, synth.BF16_NAN))
    for b, L in enumerate(w.layout.context_lens):
        t = np.arange(int(L))
        slots = w.layout.block_table[b, t // P].astype(np.int64) * P + t % P
        pa.pa_kv_write(_u16(w.k_pool[slots // P, slots % P]), _u16(w.v_pool[slots // P, slots % P]),
                       torch.from_numpy(slots).cuda(), kp, vp)
    g = gu.GqaDev(w)
    g.k, g.v = kp, vp
    o, l = g.run()
    gu.check_gqa(w, o, l)


def test_zero_tokens_is_a_no_op():
    import paged_kv_attention_19_gb300 as pa
    x = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    pool = torch.empty(1, 8, 2, 64, dtype=torch.bfloat16, device="cuda")
    pa.pa_kv_write(x, x, torch.empty(0, dtype=torch.int64, device="cuda"), pool, pool)
