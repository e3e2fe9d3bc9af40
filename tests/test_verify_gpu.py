"""Multi-query (speculative-verify) GQA decode on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import compare
import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def _run(w, num_splits=0, window=None):
    import paged_kv_attention_19_gb300 as pa
    g = gu.GqaDev(w)
    B, Q, Hq, D = w.q.shape
    out = torch.full((B, Q, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Q, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = pa.workspace_for_gqa(g.q, g.k, g.bt, num_splits)
    pa.pa_verify_gqa(g.q, g.k, g.v, g.bt, g.lens, out, lse, scale=w.scale,
                     window=w.window if window is None else window, num_splits=num_splits, workspace=ws)
    torch.cuda.synchronize()
    return gu.bits(out), lse.cpu().numpy()


def _check(w, o, l, rows=None):
    B, Q, Hq, D = w.q.shape
    ro, rl = oracle.verify_gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                               w.window, rows=rows)
    if rows is None:
        go, gl = o.reshape(-1, D), l.reshape(-1)
    else:
        idx = np.asarray(rows)
        go, gl = o[idx[:, 0], idx[:, 1], idx[:, 2]], l[idx[:, 0], idx[:, 1], idx[:, 2]]
    st = compare.compare(go, ro)
    dl = compare.lse_max_abs(gl, rl)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
    assert dl <= compare.LSE_ABS, f"lse max abs err {dl:.3e}"
    return st, dl


LADDER = [1, 2, 3, 31, 32, 33, 64, 100, 685, 1000]


@pytest.mark.parametrize("hq,hkv,D,Q", [(8, 2, 128, 2), (8, 2, 128, 5), (64, 8, 128, 2), (64, 8, 128, 4),
                                        (32, 8, 128, 7), (4, 4, 64, 16), (32, 2, 128, 3), (40, 2, 64, 2),
                                        (16, 4, 256, 3), (12, 2, 128, 4)])
def test_verify_ladder(hq, hkv, D, Q):
    w = synth.make_gqa(300 + hq + Q, LADDER, hq, hkv, D, 32, num_query=Q)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("window", [1, 7, 100])
def test_verify_window(window):
    w = synth.make_gqa(320 + window, LADDER, 8, 2, 128, 16, window=window, num_query=4)
    o, l = _run(w)
    _check(w, o, l)


@pytest.mark.parametrize("splits", [1, 3, 64, 1000])
def test_verify_splits(splits):
    w = synth.make_gqa(330 + splits, [5000, 3, 900, 0, 77], 16, 2, 128, 16, num_query=3)
    o, l = _run(w, num_splits=splits)
    _check(w, o, l)


def test_one_position_equals_decode_bitwise():
    w = synth.make_gqa(340, LADDER, 8, 2, 128, 32)
    a_o, a_l = gu.GqaDev(w).run()
    w1 = synth.GQAWorkload(**{**w.__dict__, "q": w.q[:, None], "num_query": 1})
    b_o, b_l = _run(w1)
    assert np.array_equal(a_o, b_o.reshape(a_o.shape))
    assert np.array_equal(a_l.view(np.uint32), b_l.reshape(a_l.shape).view(np.uint32))


def test_verify_scrambled_vs_identity_bitwise():
    a = synth.make_gqa(350, LADDER, 16, 2, 128, 16, num_query=3, scramble=True)
    b = synth.make_gqa(350, LADDER, 16, 2, 128, 16, num_query=3, scramble=False)
    oa, la = _run(a)
    ob, lb = _run(b)
    assert np.array_equal(oa, ob) and np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_full_size_verify_workload_every_output():
    """The full verify workload (4 query positions per qwen3-32b row) in the bench's launch
    configuration: every (row, position, head) output and LSE against the oracle."""
    w = synth.workload("qwen3-32b-verify4")
    o, l = _run(w)
    st, dl = _check(w, o, l)
    gu.report("qwen3-32b-verify4", o.shape, st, dl)
