"""FP8 (E4M3) KV cache on the GPU through the C ABI: the decode and the
multi-query verify over code pools against the fp64 oracle (codes decoded
exactly, times the per-pool scales), the quantizing write bit-exact against the
oracle's encoder, and a decode over pools the GPU wrote."""
import numpy as np
import pytest
import torch

import compare
import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

LADDER = [1, 2, 3, 31, 32, 33, 64, 100, 685, 1000]


def _run(w, num_splits=0, window=None, out=None):
    import paged_kv_attention_19_gb300 as pa
    q, k, v = gu.dev(w.q), gu.dev(w.k_pool), gu.dev(w.v_pool)
    bt, lens = gu.dev(w.layout.block_table), gu.dev(w.layout.context_lens)
    if out is None:
        out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(w.q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    ws = pa.workspace_for_gqa(q, k, bt, num_splits)
    pa.pa_decode_gqa_fp8(q, k, v, bt, lens, out, lse, scale=w.scale, k_scale=w.k_scale, v_scale=w.v_scale,
                         window=w.window if window is None else window, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return gu.bits(out), lse.cpu().numpy()


def _check(w, o, l, rows=None, window=None):
    D = w.head_dim
    ro, rl = oracle.gqa_fp8(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                            w.k_scale, w.v_scale, w.window if window is None else window, rows=rows,
                            num_query=w.num_query)
    if rows is None:
        go, gl = o.reshape(-1, D), l.reshape(-1)
    else:
        idx = np.asarray(rows)
        o4 = o.reshape(w.batch, w.num_query, w.num_q_heads, D)
        l3 = l.reshape(w.batch, w.num_query, w.num_q_heads)
        if idx.shape[1] == 2:
            idx = np.stack([idx[:, 0], np.zeros(len(idx), dtype=idx.dtype), idx[:, 1]], axis=1)
        go, gl = o4[idx[:, 0], idx[:, 1], idx[:, 2]], l3[idx[:, 0], idx[:, 1], idx[:, 2]]
    st = compare.compare(go, ro)
    dl = compare.lse_max_abs(gl, rl)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
    assert dl <= compare.LSE_ABS, f"lse max abs err {dl:.3e}"
    return st, dl


@pytest.mark.parametrize("hq,hkv,D,P", [(8, 2, 128, 32), (64, 8, 128, 32), (16, 4, 256, 32), (32, 2, 128, 16),
                                        (4, 4, 128, 8), (40, 2, 256, 64), (12, 2, 128, 256), (32, 1, 256, 16)])
def test_fp8_decode_ladder(hq, hkv, D, P):
    w = synth.make_gqa(500 + hq + D + P, LADDER, hq, hkv, D, P, fp8=True)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("window,D", [(1, 128), (7, 128), (100, 128), (333, 256)])
def test_fp8_window(window, D):
    w = synth.make_gqa(520 + window, LADDER, 8, 2, D, 16, window=window, fp8=True)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("splits", [1, 3, 152, 1000])
def test_fp8_splits(splits):
    w = synth.make_gqa(530 + splits, [5000, 3, 900, 0, 77, 4096], 16, 2, 128, 16, fp8=True)
    o, l = _run(w, num_splits=splits)
    _check(w, o, l)


@pytest.mark.parametrize("hq,hkv,D,Q,window", [(8, 2, 128, 4, 0), (64, 8, 128, 3, 0), (16, 4, 256, 5, 0),
                                               (8, 2, 128, 4, 50)])
def test_fp8_verify(hq, hkv, D, Q, window):
    w = synth.make_gqa(540 + hq + Q, LADDER, hq, hkv, D, 32, num_query=Q, window=window, fp8=True)
    o, l = _run(w)
    _check(w, o, l)


def test_fp8_scrambled_vs_identity_bitwise():
    a = synth.make_gqa(550, LADDER, 16, 2, 128, 16, fp8=True, scramble=True)
    b = synth.make_gqa(550, LADDER, 16, 2, 128, 16, fp8=True, scramble=False)
    oa, la = _run(a)
    ob, lb = _run(b)
    assert np.array_equal(oa, ob)
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_fp8_scales_are_applied():
    """The scales enter as the definition says: doubling v_scale doubles the output (exactly:
    a power of two), and k_scale multiplies the scores like the softmax scale does."""
    w = synth.make_gqa(560, LADDER, 8, 2, 128, 32, fp8=True)
    o1, l1 = _run(w)
    w2 = synth.GQAWorkload(**{**w.__dict__, "v_scale": w.v_scale * 2})
    o2, l2 = _run(w2)
    f1, f2 = synth.bf16_bits_to_f32(o1), synth.bf16_bits_to_f32(o2)
    assert np.array_equal(f2, 2 * f1)
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32))
    w3 = synth.GQAWorkload(**{**w.__dict__, "k_scale": w.k_scale * 3})
    o3, l3 = _run(w3)
    _check(w3, o3, l3)


def test_fp8_full_size_every_output():
    """The full FP8 workload in the launch configuration the benchmark times (automatic
    shares): every (row, head) output and LSE against the oracle."""
    w = synth.workload("qwen3-32b-fp8")
    o, l = _run(w)
    st, dl = _check(w, o, l)
    gu.report("qwen3-32b-fp8", o.shape, st, dl)


# ------------------------------------------------------------------------- the quantizing write
@pytest.mark.filterwarnings("ignore:overflow encountered in divide:RuntimeWarning")  # the saturating cases
@pytest.mark.parametrize("T,Hkv,D,P,pages,pad,ks,vs", [(1, 1, 16, 8, 1, 0, 1.0, 1.0),
                                                       (37, 2, 128, 16, 8, 5, 1.0, 0.5),
                                                       (300, 8, 128, 32, 16, 7, 0.37, 1.0 / 3),
                                                       (64, 4, 256, 32, 4, 0, 1.0 / 512, 2.5e-3),
                                                       (1000, 3, 64, 256, 5, 11, 3e-5, 7.0),
                                                       (50, 2, 32, 16, 4, 3, 2.0 ** -126, 2.0 ** 127),
                                                       (40, 2, 64, 16, 4, 0, 2.0 ** 126, 1e-40),
                                                       (33, 1, 16, 8, 8, 2, 0.125, 2.0 ** -9)])
def test_kv_write_fp8_bit_exact(T, Hkv, D, P, pages, pad, ks, vs):
    """Scale 1 divides exactly (the bf16 inputs hit E4M3 ties often: ties to even); 1/512 pushes
    |x| > 0.875 past 448 and 3e-5 nearly every value (saturation); 7 reaches the subnormal codes
    and zero.  Powers of two from 2^-126 to 2^126 divide as products with their reciprocal; 2^127
    (whose reciprocal is subnormal) and the subnormal scale 1e-40 take the division, and
    0.125 / 2^-9 the product, each against the oracle's float32 quotient."""
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(600 + T, T, Hkv, D, P, pages, pad_every=pad)
    kp0 = np.full(w.pool_shape(), synth.E4M3_NAN, dtype=np.uint8)
    vp0 = kp0.copy()
    ks32, vs32 = float(np.float32(ks)), float(np.float32(vs))
    ref_k, ref_v = oracle.kv_write_fp8(w.k, w.v, w.slots, kp0, vp0, ks32, vs32)
    kp, vp = gu.dev(kp0), gu.dev(vp0)
    pa.pa_kv_write_fp8(gu.dev(w.k), gu.dev(w.v), torch.from_numpy(w.slots).cuda(), kp, vp, k_scale=ks32,
                       v_scale=vs32)
    torch.cuda.synchronize()
    gk, gv = kp.cpu().numpy(), vp.cpu().numpy()
    bad = np.flatnonzero(gk.ravel() != ref_k.ravel())
    assert bad.size == 0, (bad[:8], gk.ravel()[bad[:8]], ref_k.ravel()[bad[:8]])
    assert np.array_equal(gv, ref_v)


def test_kv_write_fp8_bad_slot():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_kv_write(650, 20, 2, 64, 8, 4)
    slots = w.slots.copy()
    slots[5] = w.num_pages * w.page_size   # one past the pool
    kp0 = np.full(w.pool_shape(), synth.E4M3_NAN, dtype=np.uint8)
    ref_k, ref_v = oracle.kv_write_fp8(w.k, w.v, np.where(np.arange(20) == 5, -1, slots), kp0, kp0.copy(),
                                       0.25, 0.25)
    kp, vp = gu.dev(kp0), gu.dev(kp0.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_kv_write_fp8(gu.dev(w.k), gu.dev(w.v), torch.from_numpy(slots).cuda(), kp, vp, k_scale=0.25,
                       v_scale=0.25, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_SLOT
    assert np.array_equal(kp.cpu().numpy(), ref_k) and np.array_equal(vp.cpu().numpy(), ref_v)


def test_decode_over_gpu_written_fp8_pools():
    """Write a prefill's K/V into FP8 pools on the GPU, decode over them, and compare with the
    oracle's decode over the oracle's own quantized pools."""
    import paged_kv_attention_19_gb300 as pa
    Hq, Hkv, D, P, pages = 16, 4, 128, 16, 40
    lens = [1, 17, 200, 311]
    w = synth.make_kv_write(660, max(lens), Hkv, D, P, pages)
    ks, vs = 1.0 / 64, 1.0 / 128
    kp0 = np.full(w.pool_shape(), synth.E4M3_NAN, dtype=np.uint8)
    ref_k, ref_v = oracle.kv_write_fp8(w.k, w.v, w.slots, kp0, kp0.copy(), ks, vs)
    kp, vp = gu.dev(kp0), gu.dev(kp0.copy())
    pa.pa_kv_write_fp8(gu.dev(w.k), gu.dev(w.v), torch.from_numpy(w.slots).cuda(), kp, vp, k_scale=ks, v_scale=vs)
    # block table: row b holds tokens [sum(lens[:b]), +lens[b]) of the prefill, page-aligned
    maxp = max((L + P - 1) // P for L in lens)
    bt = np.full((len(lens), maxp), -1, dtype=np.int32)
    # row b reads the prefill's first lens[b] tokens: token t sits in page slots[t] // P
    page_of_token = (w.slots // P).astype(np.int32)
    for b, L in enumerate(lens):
        n = (L + P - 1) // P
        bt[b, :n] = page_of_token[np.arange(n) * P]
    q = synth._normal_bf16_dense(synth.stream_seed(660, synth.TAG_Q), len(lens) * Hq * D, 1.0)
    q = q.reshape(len(lens), Hq, D)
    ctx = np.asarray(lens, dtype=np.int32)
    out = torch.full((len(lens), Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((len(lens), Hq), float("nan"), dtype=torch.float32, device="cuda")
    qd, btd, ld = gu.dev(q), gu.dev(bt), gu.dev(ctx)
    ws = pa.workspace_for_gqa(qd, kp, btd)
    pa.pa_decode_gqa_fp8(qd, kp, vp, btd, ld, out, lse, scale=D ** -0.5, k_scale=ks, v_scale=vs, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(kp.cpu().numpy(), ref_k) and np.array_equal(vp.cpu().numpy(), ref_v)
    ro, rl = oracle.gqa_fp8(q, ref_k, ref_v, bt, ctx, D ** -0.5, ks, vs)
    st = compare.compare(gu.bits(out).reshape(-1, D), ro)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
    assert compare.lse_max_abs(lse.cpu().numpy().reshape(-1), rl) <= compare.LSE_ABS


def test_fp8_empty_rows_and_batch_zero():
    """Rows with no key give out = 0 and lse = -inf; batch 0 is a no-op."""
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(670, [0, 5, 0, 300], 16, 2, 128, 16, fp8=True)
    o, l = _run(w)
    _check(w, o, l)
    assert np.all(o.reshape(4, 16, 128)[[0, 2]] == 0) and np.all(np.isneginf(l.reshape(4, 16)[[0, 2]]))
    q = torch.empty(0, 16, 128, dtype=torch.bfloat16, device="cuda")
    k = gu.dev(w.k_pool)
    bt = torch.empty(0, 4, dtype=torch.int32, device="cuda")
    lens = torch.empty(0, dtype=torch.int32, device="cuda")
    out = torch.empty(0, 16, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    pa.pa_decode_gqa_fp8(q, k, k, bt, lens, out, None, scale=0.1, k_scale=1.0, v_scale=1.0, workspace=ws)
    torch.cuda.synchronize()


def test_fp8_bad_page_is_reported_not_trapped():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(680, [40, 70], 8, 2, 128, 16, fp8=True)
    q, k, v = gu.dev(w.q), gu.dev(w.k_pool), gu.dev(w.v_pool)
    lens = gu.dev(w.layout.context_lens)
    bt = w.layout.block_table.copy()
    bt[1, 2] = w.layout.num_pages + 5          # out of the pool
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pa.workspace_for_gqa(q, k, gu.dev(bt))
    pa.pa_decode_gqa_fp8(q, k, v, gu.dev(bt), lens, out, None, scale=w.scale, k_scale=w.k_scale,
                         v_scale=w.v_scale, workspace=ws)
    assert pa.pa_read_device_status(ws) & pa.PA_DEV_BAD_PAGE
    # row 0 is unaffected by row 1's bad entry
    ro, _ = oracle.gqa_fp8(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                           w.k_scale, w.v_scale, rows=[(0, h) for h in range(8)])
    assert compare.compare(gu.bits(out)[0], ro).ok()
    # a clean call clears the status word
    pa.pa_decode_gqa_fp8(q, k, v, gu.dev(w.layout.block_table), lens, out, None, scale=w.scale,
                         k_scale=w.k_scale, v_scale=w.v_scale, workspace=ws)
    assert pa.pa_read_device_status(ws) == 0


def test_fp8_run_to_run_bitwise():
    w = synth.make_gqa(690, LADDER, 64, 8, 128, 32, fp8=True)
    a = _run(w, num_splits=300)
    b = _run(w, num_splits=300)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
