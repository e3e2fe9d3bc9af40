"""pa_decode_gqa_noalloc: the GQA decode for callers that cannot allocate device
memory at call time (its workspace is a fixed array inside the library).  It must
give the results of pa_decode_gqa with a caller-provided workspace, on two calls
in a row (the second reuses the array the first one left behind), and refuse a
shape whose workspace would not fit, before launching anything.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import compare
import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu


def _noalloc(pa, g, w, out, lse, num_splits=0):
    B, Hq, D = w.q.shape
    num_pages, P, Hkv, _ = w.k_pool.shape
    max_pages = w.layout.block_table.shape[1]
    return pa.lib.pa_decode_gqa_noalloc(
        g.q.data_ptr(), g.k.data_ptr(), g.v.data_ptr(), g.bt.data_ptr(), g.lens.data_ptr(), out.data_ptr(),
        lse.data_ptr(), B, Hq, Hkv, D, P, num_pages, max_pages, max_pages * P, float(w.scale), int(w.window),
        int(num_splits), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("window", [0, 100])
def test_noalloc_matches_workspace_entry_point_twice(window):
    import paged_kv_attention_19_gb300 as pa
    w = synth.make_gqa(4242 + window, [1, 31, 32, 33, 64, 100, 685, 1000], 16, 2, 128, 32, window=window)
    g = gu.GqaDev(w)
    ref_o, ref_l = g.run()            # pa_decode_gqa with a torch-allocated workspace
    gu.check_gqa(w, ref_o, ref_l)     # and that one agrees with the oracle
    for _ in range(2):
        out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(w.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(pa, g, w, out, lse) == pa.PA_OK
        torch.cuda.synchronize()
        o, l = gu.bits(out), lse.cpu().numpy()
        st = compare.compare(o, ref_o)
        assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, str(st)
        assert compare.lse_max_abs(l, ref_l) <= compare.LSE_ABS
        assert np.isfinite(synth.bf16_bits_to_f32(o)).all()


def test_noalloc_refuses_a_workspace_larger_than_its_scratch():
    import paged_kv_attention_19_gb300 as pa
    B, Hq, Hkv, D, P, max_ctx, splits = 4, 16, 4, 256, 16, 4096, 4096
    assert pa.pa_workspace_size(pa.PA_KIND_GQA, B, Hq, Hkv, D, max_ctx, P, splits) > (32 << 20)
    x = torch.empty(16, dtype=torch.uint8, device="cuda")  # never read: the call stops on the host
    rc = pa.lib.pa_decode_gqa_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                      x.data_ptr(), None, B, Hq, Hkv, D, P, 1 << 20, max_ctx // P, max_ctx,
                                      0.1, 0, splits, torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_WORKSPACE_TOO_SMALL
