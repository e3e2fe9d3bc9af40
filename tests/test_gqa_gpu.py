"""GQA paged decode: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import compare
import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

LADDER = [1, 31, 32, 33, 64, 100, 685, 1000]
SPLITS = [1, 2, 3, 4, 5, 8, 16, 17, 64, 152, 300, 512, 4096]


def test_tiny_workload_all_rows():
    w = synth.workload("tiny")
    o, l = gu.GqaDev(w).run()
    st, dl = gu.check_gqa(w, o, l)
    assert not np.isnan(synth.bf16_bits_to_f32(o)).any()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 1), (4, 4), (16, 2), (6, 2), (24, 2), (32, 2), (40, 2), (64, 4)])
def test_context_ladder(D, hq, hkv):
    w = synth.make_gqa(100 + D + hq, LADDER, hq, hkv, D, 32, k_std=1.0)
    o, l = gu.GqaDev(w).run()
    gu.check_gqa(w, o, l)


@pytest.mark.parametrize("P", [8, 16, 64, 128, 256])
def test_page_sizes(P):
    w = synth.make_gqa(200 + P, LADDER, 8, 2, 128, P)
    o, l = gu.GqaDev(w).run()
    gu.check_gqa(w, o, l)


def test_page_size_below_eight_is_rejected():
    import paged_kv_attention_19_gb300 as pa
    assert pa.pa_workspace_size(pa.PA_KIND_GQA, 2, 8, 2, 128, 100, 4, 0) == 0
    w = synth.make_gqa(210, [40, 70], 8, 2, 128, 4)
    g = gu.GqaDev(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("window", [1, 5, 31, 32, 33, 100, 4096])
def test_window(D, window):
    w = synth.make_gqa(300 + window, LADDER, 8, 2, D, 32, window=window)
    o, l = gu.GqaDev(w).run()
    gu.check_gqa(w, o, l)


def test_window_at_least_length_is_no_window_bitwise():
    w = synth.make_gqa(333, LADDER, 8, 2, 128, 32, window=0)
    g = gu.GqaDev(w)
    a = g.run(num_splits=4)
    b = g.run(num_splits=4, window=1000)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("P", [8, 16])
@pytest.mark.parametrize("window", [0, 5, 33, 100])
def test_unit_major_stages(D, P, window):
    """Decode over pages of fewer than 32 tokens at head_dim 128 and 256 runs the kernel whose stage
    blocks are unit-major (a unit's planes filled by one 5-D copy): the ladder, with windows that
    mask stages at every offset within a unit, and several split counts."""
    w = synth.make_gqa(1100 + D + P + window, LADDER + [4096], 8, 2, D, P, window=window)
    g = gu.GqaDev(w)
    for splits in (0, 5, 64):
        o, l = g.run(num_splits=splits)
        gu.check_gqa(w, o, l)


@pytest.mark.parametrize("P", [16, 32])
def test_scrambled_vs_identity_pages_bitwise(P):
    for splits in (0, 3):
        a = synth.make_gqa(400, LADDER, 8, 2, 128, P, scramble=True)
        b = synth.make_gqa(400, LADDER, 8, 2, 128, P, scramble=False)
        assert not np.array_equal(a.layout.block_table, b.layout.block_table)
        oa, la = gu.GqaDev(a).run(num_splits=splits)
        ob, lb = gu.GqaDev(b).run(num_splits=splits)
        assert np.array_equal(oa, ob), "page order changed output bits"
        assert np.array_equal(la.view(np.uint32), lb.view(np.uint32)), "page order changed lse bits"


def test_num_splits_sweep():
    w = synth.make_gqa(500, LADDER, 8, 2, 128, 32)
    g = gu.GqaDev(w)
    ref_o, ref_l = g.run(num_splits=0)
    gu.check_gqa(w, ref_o, ref_l)
    for n in SPLITS:
        o, l = g.run(num_splits=n)
        gu.check_gqa(w, o, l)
        # different split counts agree within rounding
        st = compare.compare(o, ref_o)
        assert st.max_abs <= compare.MAX_ABS


@pytest.mark.parametrize("splits", [0, 2, 7, 64, 152, 1000])
def test_shares_spanning_rows_and_heads(splits):
    """Shares whose ranges start and end inside sequences, cover several whole sequences, or hold
    nothing; one long sequence spread over many shares; empty rows between; two 16-head subgroups."""
    w = synth.make_gqa(510 + splits, [20000, 1, 0, 3, 7000, 64, 0, 129], 40, 2, 128, 16)
    o, l = gu.GqaDev(w).run(num_splits=splits)
    gu.check_gqa(w, o, l)


def test_fewer_query_rows_than_one_tile():
    """batch * Hq below the 16 query rows one tensor-core tile holds."""
    w = synth.make_gqa(520, [77], 8, 2, 128, 16)
    o, l = gu.GqaDev(w).run()
    gu.check_gqa(w, o, l)
    w = synth.make_gqa(521, [300], 4, 1, 64, 32)
    o, l = gu.GqaDev(w).run(num_splits=3)
    gu.check_gqa(w, o, l)


def test_run_to_run_bitwise():
    w = synth.make_gqa(600, [3000, 17, 900, 4096], 32, 8, 128, 16)
    g = gu.GqaDev(w)
    first = g.run()
    for _ in range(4):
        again = g.run()
        assert np.array_equal(first[0], again[0])
        assert np.array_equal(first[1].view(np.uint32), again[1].view(np.uint32))


def test_empty_rows_and_batch_zero():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(700, [0, 5, 0, 40], 8, 2, 128, 16, extra_table_cols=1)
    for splits in (0, 1, 3):
        o, l = gu.GqaDev(w).run(num_splits=splits)
        f = synth.bf16_bits_to_f32(o)
        assert (f[0] == 0).all() and (f[2] == 0).all()
        assert np.isneginf(l[0]).all() and np.isneginf(l[2]).all()
        gu.check_gqa(w, o, l)
    # batch 0 is a no-op
    q = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    g = gu.GqaDev(w)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pa.pa_decode_gqa(q, g.k, g.v, g.bt[:0], g.lens[:0], torch.empty_like(q), None, scale=1.0, workspace=ws)


def test_lse_optional():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(710, LADDER, 8, 2, 128, 32)
    g = gu.GqaDev(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pa.workspace_for_gqa(g.q, g.k, g.bt)
    pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    o2, _ = g.run()
    assert np.array_equal(gu.bits(out), o2)


def test_bad_page_and_length_are_reported_not_trapped():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(800, [40, 70], 8, 2, 128, 16)
    g = gu.GqaDev(w)
    bt = w.layout.block_table.copy()
    bt[1, 2] = w.layout.num_pages + 5          # out of the pool
    g.bt = gu.dev(bt)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pa.workspace_for_gqa(g.q, g.k, g.bt)
    pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws)
    assert pa.pa_read_device_status(ws) & pa.PA_DEV_BAD_PAGE
    # row 0 is unaffected by row 1's bad entry
    ro, _ = gu.gqa_oracle(w, rows=[(0, h) for h in range(8)])
    assert compare.compare(gu.bits(out)[0], ro).ok()
    # a clean call clears the status word
    g.bt = gu.dev(w.layout.block_table)
    pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws)
    assert pa.pa_read_device_status(ws) == 0
    # a context length above max_context_len is clamped and reported
    lens = gu.dev(np.array([40, 70], dtype=np.int32))
    pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, lens, out, None, scale=w.scale, workspace=ws, max_context_len=64)
    assert pa.pa_read_device_status(ws) & pa.PA_DEV_BAD_LEN


def test_host_side_errors():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(900, [40, 70], 8, 2, 128, 16)
    g = gu.GqaDev(w)
    out = torch.empty(w.q.shape, dtype=torch.bfloat16, device="cuda")
    ws = pa.workspace_for_gqa(g.q, g.k, g.bt)
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_gqa(g.q, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws[: ws.numel() // 2])
    assert e.value.status == pa.PA_ERR_WORKSPACE_TOO_SMALL
    raw = torch.empty(g.q.numel() * 2 + 16, dtype=torch.uint8, device="cuda")
    qmis = raw[2: 2 + g.q.numel() * 2].view(torch.bfloat16).view(g.q.shape)   # 2-byte offset
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_gqa(qmis, g.k, g.v, g.bt, g.lens, out, None, scale=w.scale, workspace=ws)
    assert e.value.status == pa.PA_ERR_MISALIGNED


@pytest.mark.parametrize("name", ["llama3-8b", "qwen3-32b", "hd256-window"])
def test_full_size_workload_every_output(name):
    """The bench workloads at full size, in the bench's launch configuration (automatic splits):
    every (row, head) output and LSE against the oracle, with the whole-tensor statistics of the
    PR #425 numerics table (max_abs, max_rel, bitwise %, worst index)."""
    w = synth.workload(name)
    o, l = gu.GqaDev(w).run()
    st, dl = gu.check_gqa(w, o, l)
    gu.report(name, o.shape, st, dl)


@pytest.mark.parametrize("kind", ["decode", "decode-page16", "verify", "fp8", "nvfp4"])
def test_wait_limit_zero_gives_up_cleanly_and_next_call_is_clean(kind):
    """With a wait limit of 0 a CTA of the split kernel gives up at the first ring slot it finds
    busy (4 shares: every CTA streams thousands of stages, so its producer soon waits for the
    oldest one): the call returns, its status word reports PA_DEV_TIMEOUT, and (its outputs being
    unspecified) the next call at the default limit on the same workspace is clean and matches the
    oracle.  The bf16 decode (plane-major stages at page 32, unit-major at page 16), the multi-query
    verify, the FP8 kernel and the NVFP4 kernel (whose late warps keep meeting their token group's
    score-exchange barrier)."""
    import oracle
    import paged_kv_attention_19_gb300 as pa
    scales = dict(k_scale=0.25, v_scale=1.0 / 16) if kind == "nvfp4" else {}
    w = synth.make_gqa(960, LADDER + [20000] * 6, 16, 2, 128, 16 if kind == "decode-page16" else 32,
                       num_query=3 if kind == "verify" else 1,
                       fp8=kind == "fp8", nvfp4=kind == "nvfp4", **scales)
    g = gu.GqaDev(w)
    ws = pa.workspace_for_gqa(g.q, g.k, g.bt)
    try:
        pa.pa_set_wait_limit_ns(0)
        g.run_any(workspace=ws, num_splits=4)
        assert pa.pa_read_device_status(ws) & pa.PA_DEV_TIMEOUT
    finally:
        pa.pa_set_wait_limit_ns(pa.PA_DEFAULT_WAIT_LIMIT_NS)
    o, l = g.run_any(workspace=ws)
    assert pa.pa_read_device_status(ws) == 0
    lens, bt = w.layout.context_lens, w.layout.block_table
    if kind == "fp8":
        ro, rl = oracle.gqa_fp8(w.q, w.k_pool, w.v_pool, bt, lens, w.scale, w.k_scale, w.v_scale)
    elif kind == "nvfp4":
        ro, rl = oracle.gqa_nvfp4(w.q, w.k_pool, w.v_pool, bt, lens, w.scale, w.k_scale, w.v_scale)
    elif kind == "verify":
        ro, rl = oracle.verify_gqa(w.q, w.k_pool, w.v_pool, bt, lens, w.scale, w.window)
    else:
        ro, rl = gu.gqa_oracle(w)
    st = compare.compare(o.reshape(-1, w.head_dim), ro)
    assert st.ok(), str(st)
    assert compare.lse_max_abs(l.reshape(-1), rl) <= compare.LSE_ABS
