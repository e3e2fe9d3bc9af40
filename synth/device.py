"""Upload of a seeded workload to the GPU, and the binding calls that run it.

The benchmark, ``smoke()`` and the GPU tests share these helpers: they copy the
generator's arrays into torch device tensors and call the C ABI through the
package's binding.  Nothing here computes attention; the oracle comparisons
stay with the tests.
"""
from __future__ import annotations

import numpy as np


def dev(a: np.ndarray, dtype=None):
    """Device copy of a generator array (uint16 arrays are bf16 bit patterns)."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.to("cuda") if dtype is None else t.to("cuda", dtype)


def bits(t) -> np.ndarray:
    """bf16 device tensor -> host uint16 bit patterns."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class GqaDev:
    """A GQA workload (bf16 or FP8 pools, decode or verify) resident on the GPU."""

    def __init__(self, w):
        self.w = w
        self.q = dev(w.q)
        self.k = dev(w.k_pool)
        self.v = dev(w.v_pool)
        self.bt = dev(w.layout.block_table)
        self.lens = dev(w.layout.context_lens)

    def run(self, num_splits=0, window=None, out=None, lse=None, poison=True, workspace=None,
            max_context_len=None):
        """One pa_decode_gqa call (decode workloads with bf16 pools); returns (out bits, lse)."""
        import torch
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

    def run_any(self, num_splits=0, window=None, workspace=None):
        """One call of the entry point that serves the workload: pa_decode_gqa_nvfp4 for NVFP4
        pools, pa_decode_gqa_fp8 for FP8 pools, pa_verify_gqa for several query positions, else pa_decode_gqa."""
        import torch
        import paged_kv_attention_19_gb300 as pa
        w = self.w
        win = w.window if window is None else window
        out = torch.full(w.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full(w.q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
        if workspace is None:
            workspace = pa.workspace_for_gqa(self.q, self.k, self.bt, num_splits)
        if w.nvfp4:
            pa.pa_decode_gqa_nvfp4(self.q, self.k, self.v, self.bt, self.lens, out, lse, scale=w.scale,
                                   k_scale=w.k_scale, v_scale=w.v_scale, window=win, num_splits=num_splits,
                                   workspace=workspace)
        elif w.fp8:
            pa.pa_decode_gqa_fp8(self.q, self.k, self.v, self.bt, self.lens, out, lse, scale=w.scale,
                                 k_scale=w.k_scale, v_scale=w.v_scale, window=win, num_splits=num_splits,
                                 workspace=workspace)
        elif w.num_query > 1:
            pa.pa_verify_gqa(self.q, self.k, self.v, self.bt, self.lens, out, lse, scale=w.scale, window=win,
                             num_splits=num_splits, workspace=workspace)
        else:
            pa.pa_decode_gqa(self.q, self.k, self.v, self.bt, self.lens, out, lse, scale=w.scale, window=win,
                             num_splits=num_splits, workspace=workspace)
        torch.cuda.synchronize()
        return bits(out), lse.cpu().numpy()


class MlaDev:
    """An MLA absorbed workload resident on the GPU."""

    def __init__(self, w):
        self.w = w
        self.q = dev(w.q)
        self.cache = dev(w.cache)
        self.wuk = dev(w.w_uk)
        self.wuv = dev(w.w_uv)
        self.bt = dev(w.layout.block_table)
        self.lens = dev(w.layout.context_lens)

    def run(self, num_splits=0, poison=True, workspace=None):
        """One pa_decode_mla_absorbed call; returns (out bits, lse)."""
        import torch
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
