"""NVFP4 KV cache on the GPU through the C ABI: the decode and the multi-query verify over NVFP4
row pools against the fp64 oracle (E2M1 codes times E4M3 block scales times the pool scales,
decoded exactly), the quantizing write bit-exact against the oracle's quantizer, and a decode
over pools the GPU wrote."""
import numpy as np
import pytest
import torch

import compare
import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

LADDER = [1, 2, 3, 31, 32, 33, 64, 100, 685, 1000]
KS, VS = 0.25, 1.0 / 16


def _gqa(seed, lens, hq, hkv, D, P, **kw):
    kw.setdefault("k_scale", KS)
    kw.setdefault("v_scale", VS)
    return synth.make_gqa(seed, lens, hq, hkv, D, P, nvfp4=True, **kw)


def _run(w, num_splits=0, window=None):
    import paged_kv_attention_19_gb300 as pa
    q, k, v = gu.dev(w.q), gu.dev(w.k_pool), gu.dev(w.v_pool)
    bt, lens = gu.dev(w.layout.block_table), gu.dev(w.layout.context_lens)
    out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(w.q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    ws = pa.workspace_for_gqa(q, k, bt, num_splits)
    pa.pa_decode_gqa_nvfp4(q, k, v, bt, lens, out, lse, scale=w.scale, k_scale=w.k_scale, v_scale=w.v_scale,
                           window=w.window if window is None else window, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return gu.bits(out), lse.cpu().numpy()


def _check(w, o, l, rows=None):
    D = w.head_dim
    ro, rl = oracle.gqa_nvfp4(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                              w.k_scale, w.v_scale, w.window, rows=rows, num_query=w.num_query)
    if rows is None:
        go, gl = o.reshape(-1, D), l.reshape(-1)
    else:
        idx = np.asarray(rows)
        go, gl = o[idx[:, 0], idx[:, 1]], l[idx[:, 0], idx[:, 1]]
    st = compare.compare(go, ro)
    dl = compare.lse_max_abs(gl, rl)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
    assert dl <= compare.LSE_ABS, f"lse max abs err {dl:.3e}"
    return st, dl


@pytest.mark.parametrize("hq,hkv,D,P", [(8, 2, 128, 32), (64, 8, 128, 32), (16, 4, 256, 32), (32, 2, 128, 16),
                                        (4, 4, 64, 8), (40, 2, 256, 64), (12, 2, 64, 256), (32, 1, 256, 16),
                                        (8, 2, 256, 8), (16, 2, 128, 8), (20, 1, 128, 128)])
def test_nvfp4_decode_ladder(hq, hkv, D, P):
    w = _gqa(700 + hq + D + P, LADDER, hq, hkv, D, P)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("window,D", [(1, 128), (7, 64), (100, 128), (333, 256)])
def test_nvfp4_window(window, D):
    w = _gqa(720 + window, LADDER, 8, 2, D, 16, window=window)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("splits", [1, 3, 152, 1000])
def test_nvfp4_splits(splits):
    w = _gqa(730 + splits, [5000, 3, 900, 0, 77, 4096], 16, 2, 128, 16)
    o, l = _run(w, num_splits=splits)
    _check(w, o, l)


@pytest.mark.parametrize("hq,hkv,D,Q,window", [(8, 2, 128, 4, 0), (64, 8, 128, 3, 0), (16, 4, 256, 5, 0),
                                               (8, 2, 64, 4, 50)])
def test_nvfp4_verify(hq, hkv, D, Q, window):
    w = _gqa(740 + hq + Q, LADDER, hq, hkv, D, 32, num_query=Q, window=window)
    o, l = _run(w)
    _check(w, o, l)


def test_nvfp4_every_scale_code():
    """Every finite non-negative block-scale code (zero, the subnormals, up to 448) and every
    E2M1 code in the attended rows: the pools' scale bytes cycle through codes 0..126 and the
    pool scales keep the largest value (6 x 448 / 1024) small."""
    w = _gqa(750, LADDER, 16, 2, 128, 16, k_scale=2.0 ** -10, v_scale=2.0 ** -10)
    D = 128
    for pool in (w.k_pool, w.v_pool):
        sc = pool[..., D // 2: D // 2 + D // 16]
        live = sc != synth.E4M3_NAN
        cyc = (np.arange(sc.size, dtype=np.int64).reshape(sc.shape) % 127).astype(np.uint8)
        sc[live] = cyc[live]
    o, l = _run(w)
    _check(w, o, l)


def test_nvfp4_scales_are_applied():
    """Doubling v_scale doubles the output exactly (a power of two) and leaves the LSE unchanged;
    a k_scale of 3 enters the scores like the softmax scale does."""
    w = _gqa(760, LADDER, 8, 2, 128, 32)
    o1, l1 = _run(w)
    w2 = synth.GQAWorkload(**{**w.__dict__, "v_scale": w.v_scale * 2})
    o2, l2 = _run(w2)
    f1, f2 = synth.bf16_bits_to_f32(o1), synth.bf16_bits_to_f32(o2)
    assert np.array_equal(f2, 2 * f1)
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32))
    w3 = synth.GQAWorkload(**{**w.__dict__, "k_scale": w.k_scale * 3})
    o3, l3 = _run(w3)
    _check(w3, o3, l3)


def test_nvfp4_scrambled_vs_identity_bitwise():
    a = _gqa(770, LADDER, 16, 2, 128, 16, scramble=True)
    b = _gqa(770, LADDER, 16, 2, 128, 16, scramble=False)
    oa, la = _run(a)
    ob, lb = _run(b)
    assert np.array_equal(oa, ob)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_nvfp4_full_size_every_output():
    """The full NVFP4 workload in the launch configuration the benchmark times (automatic
    shares): every (row, head) output and LSE against the oracle."""
    w = synth.workload("qwen3-32b-nvfp4")
    o, l = _run(w)
    st, dl = _check(w, o, l)
    gu.report("qwen3-32b-nvfp4", o.shape, st, dl)


def test_nvfp4_empty_rows_and_bad_page():
    import paged_kv_attention_19_gb300 as pa
    w = _gqa(780, [0, 5, 0, 300], 16, 2, 128, 16)
    o, l = _run(w)
    _check(w, o, l)
    assert np.all(o.reshape(4, 16, 128)[[0, 2]] == 0) and np.all(np.isneginf(l.reshape(4, 16)[[0, 2]]))
    q, k, v = gu.dev(w.q), gu.dev(w.k_pool), gu.dev(w.v_pool)
    lens = gu.dev(w.layout.context_lens)
    bt = w.layout.block_table.copy()
    bt[3, 4] = w.layout.num_pages + 5          # out of the pool
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pa.workspace_for_gqa(q, k, gu.dev(bt))
    pa.pa_decode_gqa_nvfp4(q, k, v, gu.dev(bt), lens, out, None, scale=w.scale, k_scale=w.k_scale,
                           v_scale=w.v_scale, workspace=ws)
    assert pa.pa_read_device_status(ws) & pa.PA_DEV_BAD_PAGE
    ro, _ = oracle.gqa_nvfp4(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                             w.k_scale, w.v_scale, rows=[(1, h) for h in range(16)])
    assert compare.compare(gu.bits(out)[1], ro).ok()


def test_nvfp4_run_to_run_bitwise():
    w = _gqa(790, LADDER, 64, 8, 128, 32)
    a = _run(w, num_splits=300)
    b = _run(w, num_splits=300)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


# ------------------------------------------------------------------------- the quantizing write
def _write(w, ks, vs, slots=None, status=None):
    import paged_kv_attention_19_gb300 as pa
    T, Hkv, D = w.k.shape
    pool0 = np.full((w.num_pages, w.page_size, Hkv, synth.nvfp4_row_bytes(D)), 0xAB, dtype=np.uint8)
    kp, vp = gu.dev(pool0), gu.dev(pool0.copy())
    sl = w.slots if slots is None else slots
    pa.pa_kv_write_nvfp4(gu.dev(w.k), gu.dev(w.v), torch.from_numpy(sl).cuda(), kp, vp, k_scale=ks, v_scale=vs,
                         status=status)
    torch.cuda.synchronize()
    return pool0, kp.cpu().numpy(), vp.cpu().numpy()


@pytest.mark.filterwarnings("ignore:overflow encountered:RuntimeWarning")  # the saturating cases
@pytest.mark.parametrize("T,Hkv,D,P,pages,pad,ks,vs", [(1, 1, 64, 8, 1, 0, 1.0, 1.0),
                                                       (37, 2, 128, 16, 8, 5, 1.0, 0.5),
                                                       (300, 8, 128, 32, 16, 7, 0.37, 1.0 / 3),
                                                       (64, 4, 256, 32, 4, 0, 1.0 / 512, 2.5e-3),
                                                       (1000, 3, 64, 256, 5, 11, 3e-5, 7.0),
                                                       (50, 2, 128, 16, 4, 3, 2.0 ** -126, 2.0 ** 127),
                                                       (40, 2, 64, 16, 4, 0, 2.0 ** 126, 1e-40),
                                                       (33, 1, 256, 8, 8, 2, 0.125, 2.0 ** -9)])
def test_kv_write_nvfp4_bit_exact(T, Hkv, D, P, pages, pad, ks, vs):
    """Whole pool rows (codes, block scales, zero padding) equal the oracle's, and every other
    byte is untouched.  Scale 1 leaves the bf16 inputs on E2M1 and E4M3 ties often; 1/512 and
    3e-5 saturate the block scales at 448; 7 gives subnormal and zero block scales; the powers of
    two divide as products with their exact reciprocal, 2^127 and the subnormal 1e-40 take the
    division."""
    w = synth.make_kv_write(800 + T, T, Hkv, D, P, pages, pad_every=pad)
    ks32, vs32 = float(np.float32(ks)), float(np.float32(vs))
    pool0, gk, gv = _write(w, ks32, vs32)
    ref_k, ref_v = oracle.kv_write_nvfp4(w.k, w.v, w.slots, pool0, pool0.copy(), ks32, vs32)
    bad = np.flatnonzero(gk.ravel() != ref_k.ravel())
    assert bad.size == 0, (bad[:8], gk.ravel()[bad[:8]], ref_k.ravel()[bad[:8]])
    assert np.array_equal(gv, ref_v)


def test_kv_write_nvfp4_special_values():
    """Blocks holding NaN (scale code 0x7F, codes 0), +-inf (scale 448), -0, and all-zero blocks
    (scale code 0, codes 0), bit-exact against the oracle."""
    w = synth.make_kv_write(850, 16, 2, 64, 8, 2)
    k = w.k.copy()
    k[0, 0, 3] = 0x7FC0        # NaN in block 0 of (token 0, head 0)
    k[1, 1, 17] = 0x7F80       # +inf
    k[2, 0, 40] = 0xFF80       # -inf
    k[3, 0, :16] = 0x8000      # a block of -0
    k[4, 1, 16:32] = 0         # a block of +0
    k[5, 0, 5] = 0xFFC1        # a negative NaN
    w = synth.KVWriteWorkload(**{**w.__dict__, "k": k})
    pool0, gk, gv = _write(w, 0.5, 0.5)
    ref_k, ref_v = oracle.kv_write_nvfp4(w.k, w.v, w.slots, pool0, pool0.copy(), 0.5, 0.5)
    assert np.array_equal(gk, ref_k) and np.array_equal(gv, ref_v)


def test_kv_write_nvfp4_bad_slot():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(860, 20, 2, 64, 8, 4)
    slots = w.slots.copy()
    slots[5] = w.num_pages * w.page_size   # one past the pool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool0, gk, gv = _write(w, 0.25, 0.25, slots=slots, status=status)
    assert int(status.item()) & pa.PA_DEV_BAD_SLOT
    ref_k, ref_v = oracle.kv_write_nvfp4(w.k, w.v, np.where(np.arange(20) == 5, -1, slots), pool0, pool0.copy(),
                                         0.25, 0.25)
    assert np.array_equal(gk, ref_k) and np.array_equal(gv, ref_v)


def test_kv_write_nvfp4_full_size():
    """The benchmark's write workload (16384 tokens x 8 KV heads x head_dim 128), bit-exact."""
    w = synth.workload("kv-write-nvfp4")
    pool0, gk, gv = _write(w, w.k_scale, w.v_scale)
    ref_k, ref_v = oracle.kv_write_nvfp4(w.k, w.v, w.slots, pool0, pool0.copy(), w.k_scale, w.v_scale)
    assert np.array_equal(gk, ref_k) and np.array_equal(gv, ref_v)


def test_decode_over_gpu_written_nvfp4_pools():
    """Write a prefill's K/V into NVFP4 pools on the GPU, decode over them, and compare with the
    oracle's decode over the oracle's own quantized pools."""
    import paged_kv_attention_19_gb300 as pa
    Hq, Hkv, D, P, pages = 16, 4, 128, 16, 40
    lens = [1, 17, 200, 311]
    w = synth.make_kv_write(870, max(lens), Hkv, D, P, pages)
    ks, vs = 0.5, 0.25
    pool0, gk, gv = _write(w, ks, vs)
    ref_k, ref_v = oracle.kv_write_nvfp4(w.k, w.v, w.slots, pool0, pool0.copy(), ks, vs)
    assert np.array_equal(gk, ref_k) and np.array_equal(gv, ref_v)
    maxp = max((L + P - 1) // P for L in lens)
    bt = np.full((len(lens), maxp), -1, dtype=np.int32)
    page_of_token = (w.slots // P).astype(np.int32)
    for b, L in enumerate(lens):
        n = (L + P - 1) // P
        bt[b, :n] = page_of_token[np.arange(n) * P]
    q = synth._normal_bf16_dense(synth.stream_seed(870, synth.TAG_Q), len(lens) * Hq * D, 1.0)
    q = q.reshape(len(lens), Hq, D)
    ctx = np.asarray(lens, dtype=np.int32)
    out = torch.full((len(lens), Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((len(lens), Hq), float("nan"), dtype=torch.float32, device="cuda")
    qd, btd, ld, kp, vp = gu.dev(q), gu.dev(bt), gu.dev(ctx), gu.dev(gk), gu.dev(gv)
    ws = pa.workspace_for_gqa(qd, kp, btd)
    pa.pa_decode_gqa_nvfp4(qd, kp, vp, btd, ld, out, lse, scale=D ** -0.5, k_scale=ks, v_scale=vs, workspace=ws)
    torch.cuda.synchronize()
    ro, rl = oracle.gqa_nvfp4(q, ref_k, ref_v, bt, ctx, D ** -0.5, ks, vs)
    st = compare.compare(gu.bits(out).reshape(-1, D), ro)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
    assert compare.lse_max_abs(lse.cpu().numpy().reshape(-1), rl) <= compare.LSE_ABS
