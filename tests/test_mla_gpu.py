"""MLA absorbed decode: the CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import compare
import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [1, 3, 17, 32, 33, 128])
def test_small_all_rows(H):
    w = synth.make_mla(1000 + H, [1, 63, 64, 65, 300], H, 64)
    o, l = gu.MlaDev(w).run()
    gu.check_mla(w, o, l)


@pytest.mark.parametrize("P", [8, 16, 32, 64, 128, 256])
def test_page_sizes(P):
    w = synth.make_mla(1100 + P, [1, 31, 33, 200, 700], 8, P)
    o, l = gu.MlaDev(w).run()
    gu.check_mla(w, o, l)


def test_num_splits_sweep():
    w = synth.make_mla(1200, [1, 100, 700, 1500], 16, 64)
    g = gu.MlaDev(w)
    ref = g.run()
    for n in [1, 2, 3, 5, 17, 64, 300]:
        o, l = g.run(num_splits=n)
        gu.check_mla(w, o, l)
        assert compare.compare(o, ref[0]).max_abs <= compare.MAX_ABS


def test_scrambled_vs_identity_and_run_to_run():
    a = synth.make_mla(1300, [65, 700, 1200], 8, 64, scramble=True)
    b = synth.make_mla(1300, [65, 700, 1200], 8, 64, scramble=False)
    oa, la = gu.MlaDev(a).run(num_splits=2)
    ob, lb = gu.MlaDev(b).run(num_splits=2)
    assert np.array_equal(oa, ob) and np.array_equal(la.view(np.uint32), lb.view(np.uint32))
    for _ in range(3):
        oc, lc = gu.MlaDev(a).run(num_splits=2)
        assert np.array_equal(oa, oc) and np.array_equal(la.view(np.uint32), lc.view(np.uint32))


def test_empty_row():
    w = synth.make_mla(1400, [0, 70], 4, 64)
    o, l = gu.MlaDev(w).run()
    assert (synth.bf16_bits_to_f32(o)[0] == 0).all() and np.isneginf(l[0]).all()
    gu.check_mla(w, o, l)


def test_full_size_workload_every_output():
    """The full MLA workload in the bench's launch configuration: every (row, head) output and
    LSE against the oracle."""
    w = synth.workload("mla")
    o, l = gu.MlaDev(w).run()
    st, dl = gu.check_mla(w, o, l)
    gu.report("mla", o.shape, st, dl)


@pytest.mark.parametrize("H", [200, 256])
def test_several_head_tiles(H):
    """More than 128 heads: two tiles of the tensor-core core (the second one partial for H = 200),
    automatic and explicit split counts."""
    w = synth.make_mla(1500 + H, [1, 65, 300, 700], H, 64)
    g = gu.MlaDev(w)
    for n in [0, 3]:
        o, l = g.run(num_splits=n)
        gu.check_mla(w, o, l)


def test_bad_page_is_reported_not_trapped():
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_mla(1600, [70, 200], 16, 64)
    g = gu.MlaDev(w)
    bt = w.layout.block_table.copy()
    bt[1, 2] = w.layout.num_pages + 5          # out of the pool
    g.bt = gu.dev(bt)
    ws = pa.workspace_for_mla(g.q, g.cache, g.bt, 0)
    o, l = g.run(workspace=ws)
    assert pa.pa_read_device_status(ws) & pa.PA_DEV_BAD_PAGE
    # row 0 is unaffected by row 1's bad entry
    gu.check_mla(w, o, l, rows=[(0, h) for h in range(16)])
    # a clean call clears the status word
    g.bt = gu.dev(w.layout.block_table)
    o, l = g.run(workspace=ws)
    assert pa.pa_read_device_status(ws) == 0
    gu.check_mla(w, o, l)
