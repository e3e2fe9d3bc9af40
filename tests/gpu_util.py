"""Helpers of the GPU parity tests: upload a seeded workload, run the CUDA path
through the C ABI binding, and compare with the fp64 oracle (imported only by
the comparison helpers, so the benchmark can reuse the upload helpers)."""
from __future__ import annotations

import numpy as np
import torch

import compare
import synth


def dev(a: np.ndarray, dtype=None):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to("cuda") if dtype is None else t.to("cuda", dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class GqaDev:
    """A GQA workload resident on the GPU."""

    def __init__(self, w: synth.GQAWorkload):
        self.w = w
        self.q = dev(w.q)
        self.k = dev(w.k_pool)
        self.v = dev(w.v_pool)
        self.bt = dev(w.layout.block_table)
        self.lens = dev(w.layout.context_lens)

    def run(self, num_splits=0, window=None, out=None, lse=None, poison=True, workspace=None,
            max_context_len=None):
        import paged_kv_attention_19_gb300 as pa
        w = self.w
        B, Hq, D = w.q.shape
        if out is None:
            out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
            if poison:
                out.fill_(float("nan"))
        if lse is None:
            lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
        if workspace is None:
            workspace = pa.workspace_for_gqa(self.q, self.k, self.bt, num_splits, max_context_len)
        pa.pa_decode_gqa(self.q, self.k, self.v, self.bt, self.lens, out, lse, scale=w.scale,
                         window=w.window if window is None else window, num_splits=num_splits,
                         workspace=workspace, max_context_len=max_context_len)
        torch.cuda.synchronize()
        return bits(out), lse.cpu().numpy()


def gqa_oracle(w: synth.GQAWorkload, rows=None, window=None):
    import oracle
    return oracle.gqa(w.q, w.k_pool, w.v_pool, w.layout.block_table, w.layout.context_lens, w.scale,
                      w.window if window is None else window, rows=rows)


def check_gqa(w, out_bits, lse, rows=None, window=None, tol_abs=compare.MAX_ABS, tol_rel=compare.MAX_REL):
    """Compare GPU output (all rows, or the sampled (b, h) rows) with the oracle; return stats."""
    B, Hq, D = w.q.shape
    ro, rl = gqa_oracle(w, rows, window)
    if rows is None:
        got_o = out_bits.reshape(-1, D)
        got_l = lse.reshape(-1)
    else:
        idx = np.asarray(rows)
        got_o = out_bits[idx[:, 0], idx[:, 1]]
        got_l = lse[idx[:, 0], idx[:, 1]]
    st = compare.compare(got_o, ro)
    dl = compare.lse_max_abs(got_l, rl)
    assert st.max_abs <= tol_abs and st.max_rel <= tol_rel, f"{w.name}: {st}"
    assert dl <= compare.LSE_ABS, f"{w.name}: lse max abs err {dl:.3e}"
    return st, dl


class MlaDev:
    def __init__(self, w: synth.MLAWorkload):
        self.w = w
        self.q = dev(w.q)
        self.cache = dev(w.cache)
        self.wuk = dev(w.w_uk)
        self.wuv = dev(w.w_uv)
        self.bt = dev(w.layout.block_table)
        self.lens = dev(w.layout.context_lens)

    def run(self, num_splits=0, poison=True, workspace=None):
        import paged_kv_attention_19_gb300 as pa
        w = self.w
        B, H, _ = w.q.shape
        out = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
        if poison:
            out.fill_(float("nan"))
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        if workspace is None:
            workspace = pa.workspace_for_mla(self.q, self.cache, self.bt, num_splits)
        pa.pa_decode_mla_absorbed(self.q, self.cache, self.wuk, self.wuv, self.bt, self.lens, out, lse,
                                  scale=w.scale, num_splits=num_splits, workspace=workspace)
        torch.cuda.synchronize()
        return bits(out), lse.cpu().numpy()


def check_mla(w, out_bits, lse, rows=None):
    import oracle
    B, H, _ = w.q.shape
    ro, rl = oracle.mla(w.q, w.cache, w.w_uk, w.w_uv, w.layout.block_table, w.layout.context_lens, w.scale,
                        rows=rows)
    if rows is None:
        got_o = out_bits.reshape(-1, 128)
        got_l = lse.reshape(-1)
    else:
        idx = np.asarray(rows)
        got_o = out_bits[idx[:, 0], idx[:, 1]]
        got_l = lse[idx[:, 0], idx[:, 1]]
    st = compare.compare(got_o, ro)
    dl = compare.lse_max_abs(got_l, rl)
    assert st.max_abs <= compare.MAX_ABS and st.max_rel <= compare.MAX_REL, f"{w.name}: {st}"
    assert dl <= compare.LSE_ABS, f"{w.name}: lse max abs err {dl:.3e}"
    return st, dl


def sample_rows(B, H, n, seed):
    u = synth.uniform01(seed, np.arange(2 * n, dtype=np.uint64))
    b = np.minimum((u[:n] * B).astype(np.int64), B - 1)
    h = np.minimum((u[n:] * H).astype(np.int64), H - 1)
    return [(int(x), int(y)) for x, y in zip(b, h)]
