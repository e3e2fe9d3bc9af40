"""Independent references that pin the fp64 oracle (test code only).

They share nothing with the oracle's C loops: the KV data are regenerated
from the generator's counter definition (logical row / token / head / dim,
never through the block table or the pool), and the arithmetic is dense
torch float64 (matmul, softmax, logsumexp, einsum).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import synth


def _logical_pool_rows(seed: int, tag: int, layout: synth.PagedLayout, b: int, width: int,
                       std: float) -> np.ndarray:
    """Row b's tokens [ceil(L/P) * P, width] as float64, drawn from the stream by logical index."""
    P = layout.page_size
    L = int(layout.context_lens[b])
    n_pages = (L + P - 1) // P
    per_page = P * width
    g0 = int(layout.logical_page_of_row[b])
    idx = np.arange(g0 * per_page, (g0 + n_pages) * per_page, dtype=np.uint64)
    vals = synth.normal_bf16(synth.stream_seed(seed, tag), idx, std)
    return synth.bf16_bits_to_f32(vals).astype(np.float64).reshape(n_pages * P, width)


def dense_gqa(w: synth.GQAWorkload, window=None):
    """softmax(q K^T scale) V per (b, h) over the visible keys; returns o [B, Hq, D], lse [B, Hq]."""
    window = w.window if window is None else window
    B, Hq, D = w.q.shape
    Hkv = w.num_kv_heads
    G = Hq // Hkv
    q = torch.from_numpy(synth.bf16_bits_to_f32(w.q).astype(np.float64))
    o = torch.zeros(B, Hq, D, dtype=torch.float64)
    lse = torch.full((B, Hq), -math.inf, dtype=torch.float64)
    for b in range(B):
        L = int(w.layout.context_lens[b])
        lo, hi = synth.visible_range(L, window)
        if hi <= lo:
            continue
        K = _logical_pool_rows(w.seed, synth.TAG_K, w.layout, b, Hkv * D, w.k_std)[lo:hi]
        V = _logical_pool_rows(w.seed, synth.TAG_V, w.layout, b, Hkv * D, 1.0)[lo:hi]
        K = torch.from_numpy(K).reshape(hi - lo, Hkv, D)
        V = torch.from_numpy(V).reshape(hi - lo, Hkv, D)
        for h in range(Hq):
            s = (K[:, h // G, :] @ q[b, h]) * w.scale
            o[b, h] = torch.softmax(s, dim=0) @ V[:, h // G, :]
            lse[b, h] = torch.logsumexp(s, dim=0)
    return o.numpy(), lse.numpy()


def dense_verify(w: synth.GQAWorkload):
    """Causal multi-query attention in dense torch float64: the row's Q newest tokens are the
    queries; a [Q, T] mask lets query i see key t when t <= L - Q + i (and t > L - Q + i - W
    under a window).  Returns o [B, Q, Hq, D], lse [B, Q, Hq]."""
    B, Q, Hq, D = w.q.shape
    Hkv = w.num_kv_heads
    G = Hq // Hkv
    q = torch.from_numpy(synth.bf16_bits_to_f32(w.q).astype(np.float64))
    o = torch.zeros(B, Q, Hq, D, dtype=torch.float64)
    lse = torch.full((B, Q, Hq), -math.inf, dtype=torch.float64)
    for b in range(B):
        L = int(w.layout.context_lens[b])
        if L == 0:
            continue
        K = torch.from_numpy(_logical_pool_rows(w.seed, synth.TAG_K, w.layout, b, Hkv * D, w.k_std)[:L])
        V = torch.from_numpy(_logical_pool_rows(w.seed, synth.TAG_V, w.layout, b, Hkv * D, 1.0)[:L])
        K, V = K.reshape(L, Hkv, D), V.reshape(L, Hkv, D)
        t = torch.arange(L)
        pos = L - Q + torch.arange(Q)                       # logical position of each query
        see = t[None, :] <= pos[:, None]
        if w.window > 0:
            see &= t[None, :] > pos[:, None] - w.window
        for h in range(Hq):
            s = (q[b, :, h, :] @ K[:, h // G, :].T) * w.scale  # [Q, L]
            s = s.masked_fill(~see, -math.inf)
            for i in range(Q):
                if see[i].any():
                    o[b, i, h] = torch.softmax(s[i], dim=0) @ V[:, h // G, :]
                    lse[b, i, h] = torch.logsumexp(s[i], dim=0)
    return o.numpy(), lse.numpy()


def logical_cache(w: synth.MLAWorkload, b: int) -> np.ndarray:
    L = int(w.layout.context_lens[b])
    return _logical_pool_rows(w.seed, synth.TAG_CACHE, w.layout, b, synth.MLA_CDIM, 1.0)[:L]


def _mla_tensors(w: synth.MLAWorkload):
    f = lambda a: torch.from_numpy(synth.bf16_bits_to_f32(a).astype(np.float64))
    return f(w.q), f(w.w_uk), f(w.w_uv)


def dense_mla_absorbed(w: synth.MLAWorkload, rows):
    """Absorbed form: q_lat = W_UK^T q_nope, attend over the 576-wide cache, o = W_UV o_lat."""
    q, wuk, wuv = _mla_tensors(w)
    out_o, out_lse = [], []
    cache_rows = {}
    for b, h in rows:
        if b not in cache_rows:
            cache_rows[b] = torch.from_numpy(logical_cache(w, b))
        C = cache_rows[b]
        q_nope, q_rope = q[b, h, :128], q[b, h, 128:]
        q_lat = torch.einsum("d,dj->j", q_nope, wuk[h])
        s = (C[:, :512] @ q_lat + C[:, 512:] @ q_rope) * w.scale
        p = torch.softmax(s, dim=0)
        o_lat = p @ C[:, :512]
        out_o.append(torch.einsum("vj,j->v", wuv[h], o_lat))
        out_lse.append(torch.logsumexp(s, dim=0))
    return torch.stack(out_o).numpy(), torch.stack(out_lse).numpy()


def dense_mla_unabsorbed(w: synth.MLAWorkload, rows):
    """Unabsorbed form: materialise per-head keys K_nope = W_UK c_lat and values V = W_UV c_lat,
    then plain multi-head attention over [q_nope || q_rope] . [K_nope || c_rope]."""
    q, wuk, wuv = _mla_tensors(w)
    out_o, out_lse = [], []
    for b, h in rows:
        C = torch.from_numpy(logical_cache(w, b))
        k_nope = torch.einsum("dj,tj->td", wuk[h], C[:, :512])     # [L, 128]
        vals = torch.einsum("vj,tj->tv", wuv[h], C[:, :512])       # [L, 128]
        keys = torch.cat([k_nope, C[:, 512:]], dim=1)              # [L, 192]
        s = (keys @ q[b, h]) * w.scale
        out_o.append(torch.softmax(s, dim=0) @ vals)
        out_lse.append(torch.logsumexp(s, dim=0))
    return torch.stack(out_o).numpy(), torch.stack(out_lse).numpy()
