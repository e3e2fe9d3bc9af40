"""pa_decode_gqa_noalloc: the GQA decode for callers that cannot allocate device
memory at call time (its workspace is a fixed array inside the library).  It must
give the results of pa_decode_gqa with a caller-provided workspace, bit for bit
(both launch the same kernels with the same share count), on two calls in a row
(the second reuses the array the first one left behind), and refuse a shape whose
workspace would not fit, before launching anything.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 32 << 20  # PA_NOALLOC_SCRATCH_BYTES


def _noalloc(pa, g, w, out, lse, num_splits=0):
    B, Hq, D = w.q.shape
    num_pages, P, Hkv, _ = w.k_pool.shape
    max_pages = w.layout.block_table.shape[1]
    return pa.lib.pa_decode_gqa_noalloc(
        g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.bt.data_ptr(), g.lens.data_ptr(), out.data_ptr(),
        lse.data_ptr(), B, Hq, Hkv, D, P, num_pages, max_pages, max_pages * P, float(w.scale), int(w.window),
        int(num_splits), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("window,num_splits", [(0, 0), (100, 0), (0, 960)])
def test_noalloc_matches_workspace_entry_point_twice(window, num_splits):
    """Automatic shares, a window, and 960 explicit shares: a workspace of about 31.7 MB of the
    33.5 MB array, so the last shares' partials sit near its top."""
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(4242 + window, [1, 31, 32, 33, 64, 100, 685, 1000, 5000, 20000], 16, 2, 128, 32,
                       window=window)
    B, Hq, D = w.q.shape
    need = pa.pa_workspace_size(pa.PA_KIND_GQA, B, Hq, 2, D, w.layout.block_table.shape[1] * 32, 32, num_splits)
    assert 0 < need <= NOALLOC_BYTES
    if num_splits:
        assert need > NOALLOC_BYTES - (2 << 20)
    g = gu.GqaDev(w)
    ref_o, ref_l = g.run(num_splits=num_splits)  # pa_decode_gqa with a torch-allocated workspace
    gu.check_gqa(w, ref_o, ref_l)                # and that one agrees with the oracle
    for _ in range(2):
        out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(pa, g, w, out, lse, num_splits) == pa.PA_OK
        torch.cuda.synchronize()
        o, l = gu.bits(out), lse.cpu().numpy()
        assert np.array_equal(o, ref_o), "output bits differ from pa_decode_gqa"
        assert np.array_equal(l.view(np.uint32), ref_l.view(np.uint32)), "lse bits differ from pa_decode_gqa"


@pytest.mark.parametrize("num_splits", [600, 4096])
def test_noalloc_refuses_a_workspace_larger_than_its_scratch(num_splits):
    """A valid small workload (head_dim 256, pools sized to its pages) whose share count needs more
    than the array: refused before any device work, outputs untouched.  Were the size check ever
    lost, the regular entry point's own workspace check would still stop the call, and every
    pointer here is a real buffer of the declared shape."""
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(4300 + num_splits, [40, 700, 3], 8, 2, 256, 16)
    B, Hq, D = w.q.shape
    need = pa.pa_workspace_size(pa.PA_KIND_GQA, B, Hq, 2, D, w.layout.block_table.shape[1] * 16, 16, num_splits)
    assert need > NOALLOC_BYTES
    g = gu.GqaDev(w)
    out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    assert _noalloc(pa, g, w, out, lse, num_splits) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    # the same call within the array's size works
    assert _noalloc(pa, g, w, out, lse, 0) == pa.PA_OK
    torch.cuda.synchronize()
    gu.check_gqa(w, gu.bits(out), lse.cpu().numpy())
