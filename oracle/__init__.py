"""fp64 CPU oracle for paged decode attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package.  The product path (the CUDA library and its
Python binding) never does, and this package never imports the product.

The arithmetic lives in ``pa_oracle.c`` (plain loops in double, OpenMP over
independent (row, head) items).  This module only compiles it, marshals numpy
arrays and converts error codes.  Each function documents which passage of
the pages it follows; the C file has the full list of readings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (-O2, OpenMP) into oracle/_build/libpa_oracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.pa_oracle_gqa.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, D, I, I, P, P, P, P, I]
    lib.pa_oracle_gqa_span.argtypes = [P, P, P, P, I, I, I, I, I, I, I, D, I, P, P, P, P, P, P, I]
    lib.pa_oracle_merge.argtypes = [I, I, P, P, P, P]
    lib.pa_oracle_mla.argtypes = [P, P, P, P, P, P, I, I, I, I, I, D, I, P, P, P, P, P, P, I]
    lib.pa_oracle_num_threads.argtypes = []
    for f in ("pa_oracle_gqa", "pa_oracle_gqa_span", "pa_oracle_merge", "pa_oracle_mla",
              "pa_oracle_num_threads"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def num_threads(lib=None) -> int:
    return int(_load(lib).pa_oracle_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _items(B, H, rows):
    if rows is None:
        bb, hh = np.meshgrid(np.arange(B), np.arange(H), indexing="ij")
        return _c(bb.ravel(), np.int32), _c(hh.ravel(), np.int32)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    return _c(rows[:, 0], np.int32), _c(rows[:, 1], np.int32)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its inputs (code {rc})")


def gqa(q, k_pool, v_pool, block_table, context_lens, scale: float, window: int = 0,
        rows=None, threads: int = 0, lib=None):
    """GQA paged decode in fp64.

    q [B, Hq, D], pools [pages, P, Hkv, D] (bf16 bit patterns, uint16), block_table
    [B, max_pages] int32, context_lens [B] int32.  ``rows``: optional list of (b, h)
    pairs; default all.  Returns (o [n, D] float64, lse [n] float64).
    Query head h reads KV head h // (Hq // Hkv); with window W > 0 a row of length
    L attends to its W most recent keys.
    """
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    bt, lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B, Hq, D = q.shape
    npg, P, Hkv, D2 = k_pool.shape
    assert D2 == D and v_pool.shape == k_pool.shape and bt.shape[0] == B
    ib, ih = _items(B, Hq, rows)
    n = ib.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _load(lib).pa_oracle_gqa(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt), _ptr(lens), B, Hq,
                               Hkv, D, P, npg, bt.shape[1], float(scale), int(window), n,
                               _ptr(ib), _ptr(ih), _ptr(o), _ptr(lse), int(threads))
    _check(rc, "gqa")
    return o, lse


def verify_gqa(q, k_pool, v_pool, block_table, context_lens, scale: float, window: int = 0,
               rows=None, threads: int = 0, lib=None):
    """Multi-query (speculative-verify) GQA decode: q [B, Q, Hq, D] holds the Q newest tokens of
    each row, so query position i of a row of length L sits at logical position L - Q + i and
    attends to the keys up to and including its own (the W most recent of them under a window):
    exactly the decode of a row of length L - Q + 1 + i (kernel-matrix row
    KERNEL-ATTN-DFLASH-PAGED-BLOCK, causal within the block; pegainfer PR #938's verify path).
    The oracle is that definition written out: every (row, position) becomes a decode row with
    its own length over the same block table.  ``rows``: optional (b, i, h) triples.  Returns
    (o [n, D], lse [n]) in (b, i, h) order."""
    q = _c(q, np.uint16)
    B, Q, Hq, D = q.shape
    bt, lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    qv = q.reshape(B * Q, Hq, D)
    btv = np.repeat(bt, Q, axis=0)
    lensv = np.maximum(np.repeat(lens, Q) - Q + 1 + np.tile(np.arange(Q, dtype=np.int32), B), 0).astype(np.int32)
    rv = None if rows is None else [(b * Q + i, h) for b, i, h in rows]
    return gqa(qv, k_pool, v_pool, btv, lensv, scale, window, rows=rv, threads=threads, lib=lib)


def gqa_span(q, k_pool, v_pool, block_table, scale: float, items, threads: int = 0, lib=None):
    """Attention of (b, h) over the explicit logical token span [t0, t1): items = [(b, h, t0, t1)]."""
    q, k_pool, v_pool = _c(q, np.uint16), _c(k_pool, np.uint16), _c(v_pool, np.uint16)
    bt = _c(block_table, np.int32)
    B, Hq, D = q.shape
    npg, P, Hkv, _ = k_pool.shape
    it = np.asarray(items, dtype=np.int64).reshape(-1, 4)
    ib, ih = _c(it[:, 0], np.int32), _c(it[:, 1], np.int32)
    t0, t1 = _c(it[:, 2], np.int64), _c(it[:, 3], np.int64)
    n = it.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    rc = _load(lib).pa_oracle_gqa_span(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt), B, Hq, Hkv, D, P,
                                    npg, bt.shape[1], float(scale), n, _ptr(ib), _ptr(ih), _ptr(t0),
                                    _ptr(t1), _ptr(o), _ptr(lse), int(threads))
    _check(rc, "gqa_span")
    return o, lse


def merge(parts_o, parts_lse, lib=None):
    """LSE merge of split partials in ascending split order; empty splits carry lse = -inf."""
    po = _c(parts_o, np.float64)
    pl = _c(parts_lse, np.float64)
    n, D = po.shape
    o = np.zeros(D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(_load(lib).pa_oracle_merge(n, D, _ptr(po), _ptr(pl), _ptr(o), _ptr(lse)), "merge")
    return o, float(lse[0])


def mla(q, cache, w_uk, w_uv, block_table, context_lens, scale: float, rows=None,
        threads: int = 0, intermediates: bool = False, lib=None):
    """MLA absorbed decode in fp64 (the seven steps of the absorbed schedule, no bf16 landings).

    q [B, H, 192] (nope 128 || rope 64), cache [pages, P, 576], w_uk / w_uv [H, 128, 512].
    Returns (o [n, 128], lse [n]) and, with ``intermediates``, also (q_lat [n, 512], o_lat [n, 512]).
    """
    q, cache = _c(q, np.uint16), _c(cache, np.uint16)
    w_uk, w_uv = _c(w_uk, np.uint16), _c(w_uv, np.uint16)
    bt, lens = _c(block_table, np.int32), _c(context_lens, np.int32)
    B, H, QD = q.shape
    npg, P, CD = cache.shape
    assert QD == 192 and CD == 576 and w_uk.shape == (H, 128, 512) and w_uv.shape == (H, 128, 512)
    ib, ih = _items(B, H, rows)
    n = ib.shape[0]
    o = np.zeros((n, 128), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    ql = np.zeros((n, 512), dtype=np.float64) if intermediates else None
    ol = np.zeros((n, 512), dtype=np.float64) if intermediates else None
    rc = _load(lib).pa_oracle_mla(_ptr(q), _ptr(cache), _ptr(w_uk), _ptr(w_uv), _ptr(bt), _ptr(lens), B, H,
                               P, npg, bt.shape[1], float(scale), n, _ptr(ib), _ptr(ih), _ptr(o),
                               _ptr(lse), _ptr(ql) if ql is not None else None,
                               _ptr(ol) if ol is not None else None, int(threads))
    _check(rc, "mla")
    if intermediates:
        return o, lse, ql, ol
    return o, lse


def kv_write(k, v, slots, k_pool, v_pool):
    """Paged KV write (vllm.cpp kernel-matrix, row KERNEL-KV-CACHE, ReshapeAndCache): for every
    token t with slot s = slots[t] >= 0, the row of physical page s // P, position s % P of each
    pool becomes token t's row.  Negative slots are padding.  Returns new pools (inputs untouched);
    bit patterns are copied, so the result is exact."""
    kp, vp = k_pool.copy(), v_pool.copy()
    P = kp.shape[1]
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        kp[s // P, s % P] = k[t]
        vp[s // P, s % P] = v[t]
    return kp, vp


def mla_cache_write(c_lat, k_rope, slots, cache):
    """MLA cache write (same row, ConcatAndCacheMla): the 576-wide row of token t is its 512
    latent values followed by its 64 rope-key values."""
    out = cache.copy()
    P = out.shape[1]
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        out[s // P, s % P, :512] = c_lat[t]
        out[s // P, s % P, 512:] = k_rope[t]
    return out


# ----------------------------------------------------------------------------- FP8 (E4M3) KV cache
# The quantized KV cache of the vllm.cpp kernel-matrix row KERNEL-KV-QUANT ("FP8"), read as: the
# pools hold FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
# infinities; S.1111.111 is NaN; largest finite magnitude 448), and one float scale per pool
# turns a code into its value: K = decode(code) * k_scale, V = decode(code) * v_scale.

def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (float64), from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return s * val


_E4M3_POS = e4m3_decode(np.arange(127, dtype=np.uint8))  # finite non-negative codes 0..126, ascending


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each value: round to nearest, ties to the code with an even
    mantissa, magnitudes above 448 saturate to 448, NaN maps to the NaN code (the saturating
    conversion of the write step)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    idx = np.searchsorted(_E4M3_POS, np.minimum(a, 448.0))      # first code >= a
    hi = np.minimum(idx, 126)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - np.minimum(a, 448.0)
    d_lo = np.minimum(a, 448.0) - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0))
    code = np.where(pick_lo, lo, hi)
    code = np.where(a >= 448.0, 126, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def kv_write_fp8(k, v, slots, k_pool, v_pool, k_scale: float, v_scale: float):
    """FP8 paged KV write: token t's bf16 rows k[t], v[t] are divided by the pool's scale in
    float32 and stored as E4M3 codes at slot slots[t] (negative: padding).  Returns new pools."""
    kf = synth_bf16_to_f32(k) / np.float32(k_scale)
    vf = synth_bf16_to_f32(v) / np.float32(v_scale)
    return kv_write(e4m3_encode(kf.astype(np.float64)), e4m3_encode(vf.astype(np.float64)), slots, k_pool, v_pool)


# ---------------------------------------------------------------------------------------------
# NVFP4 KV cache (vllm.cpp kernel-matrix, row KERNEL-KV-QUANT: "Quantized KV cache, including FP8
# and NVFP4").  The pages name the format only; this is the published NVFP4 layout read plainly:
# 4-bit E2M1 values (1 sign, 2 exponent, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6),
# one E4M3 scale per block of 16 consecutive values, and one fp32 scale per pool, so that
# value = e2m1(code) * e4m3(block scale) * pool_scale.  A pool row (page slot, KV head) of D
# values is D / 2 bytes of code pairs (the even dim in the low nibble), then D / 16 scale codes,
# then zero bytes up to a multiple of 16 bytes (nvfp4_row_bytes).

_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def nvfp4_row_bytes(D: int) -> int:
    """Bytes of one NVFP4 pool row of D values: codes and block scales, padded to 16 bytes."""
    return (D // 2 + D // 16 + 15) // 16 * 16


def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (float64), from the format's definition: exponent e, mantissa
    m; e = 0: m / 2 (subnormal), else (1 + m / 2) * 2^(e - 1); bit 3 the sign."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 15
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    val = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1))
    return np.where(c >> 3, -val, val)


def e2m1_encode(y) -> np.ndarray:
    """Nearest E2M1 code of each value: round to nearest, ties to the code with an even mantissa,
    magnitudes above 6 saturate to 6, NaN maps to +0 (E2M1 has no NaN; a NaN input also makes its
    block's scale NaN)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(np.nan_to_num(y, nan=0.0)), 6.0)
    idx = np.searchsorted(_E2M1_MAG, a)                        # first magnitude >= a
    hi = np.minimum(idx, 7)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E2M1_MAG[hi] - a
    d_lo = a - _E2M1_MAG[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((lo & 1) == 0))
    code = np.where(pick_lo, lo, hi)
    code = code | np.where(np.signbit(y) & ~np.isnan(y), 8, 0)
    return code.astype(np.uint8)


def nvfp4_quantize_rows(x32, pool_scale: float):
    """NVFP4 codes and block scales of float32 rows x32 [..., D] (D a multiple of 16), in float32
    arithmetic, each step correctly rounded: per block of 16, its amax a, the scale code
    e4m3((a / pool_scale) / 6); each value's code e2m1((x / pool_scale) / e4m3(scale)), all codes 0
    where the scale decodes to 0.  Returns (codes [..., D] uint8 (one per value), scales [..., D / 16])."""
    x = np.asarray(x32, dtype=np.float32)
    D = x.shape[-1]
    blocks = x.reshape(x.shape[:-1] + (D // 16, 16))
    ps = np.float32(pool_scale)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        a = np.max(np.abs(blocks), axis=-1)
        t = (a / ps) / np.float32(6.0)
        sc = e4m3_encode(t.astype(np.float64))
        ds = e4m3_decode(sc).astype(np.float32)
        y = (blocks / ps) / ds[..., None]
    codes = e2m1_encode(y.astype(np.float64))
    codes = np.where((ds == 0)[..., None], np.uint8(0), codes)
    return codes.reshape(x.shape), sc


def nvfp4_pack_rows(codes, scales) -> np.ndarray:
    """Pool rows [..., nvfp4_row_bytes(D)] from per-value codes [..., D] and scales [..., D / 16]."""
    codes = np.asarray(codes, dtype=np.uint8)
    D = codes.shape[-1]
    R = nvfp4_row_bytes(D)
    out = np.zeros(codes.shape[:-1] + (R,), dtype=np.uint8)
    out[..., : D // 2] = (codes[..., 0::2] & 15) | ((codes[..., 1::2] & 15) << 4)
    out[..., D // 2: D // 2 + D // 16] = scales
    return out


def nvfp4_decode_rows(rows, D: int, pool_scale: float) -> np.ndarray:
    """Values (float64 [..., D]) of NVFP4 pool rows: e2m1(code) * e4m3(block scale) * pool_scale."""
    r = np.asarray(rows, dtype=np.uint8)
    pairs = r[..., : D // 2]
    codes = np.stack([pairs & 15, pairs >> 4], axis=-1).reshape(r.shape[:-1] + (D,))
    sc = e4m3_decode(r[..., D // 2: D // 2 + D // 16])
    v = e2m1_decode(codes).reshape(r.shape[:-1] + (D // 16, 16)) * sc[..., None]
    return v.reshape(r.shape[:-1] + (D,)) * float(np.float32(pool_scale))


def kv_write_nvfp4(k, v, slots, k_pool, v_pool, k_scale: float, v_scale: float):
    """NVFP4 paged KV write: token t's bf16 rows k[t], v[t] ([T, Hkv, D]) are quantized per KV
    head (nvfp4_quantize_rows) and stored as pool rows at slot slots[t] (negative: padding).
    Returns new pools ([num_pages, P, Hkv, nvfp4_row_bytes(D)])."""
    kq = nvfp4_pack_rows(*nvfp4_quantize_rows(synth_bf16_to_f32(k), k_scale))
    vq = nvfp4_pack_rows(*nvfp4_quantize_rows(synth_bf16_to_f32(v), v_scale))
    return kv_write(kq, vq, slots, k_pool, v_pool)


def gqa_nvfp4(q, k_rows, v_rows, block_table, context_lens, scale: float, k_scale: float, v_scale: float,
              window: int = 0, rows=None, num_query: int = 1):
    """GQA decode (or multi-query verify) over an NVFP4 cache, in float64: the attention of the
    decode oracle with keys and values nvfp4_decode_rows of their pool rows.  Returns
    (o [n, D], lse [n])."""
    q = np.asarray(q, dtype=np.uint16)
    D = q.shape[-1]
    K = nvfp4_decode_rows(k_rows, D, k_scale)
    V = nvfp4_decode_rows(v_rows, D, v_scale)
    return _gqa_dense_values(q, K, V, block_table, context_lens, scale, window, rows, num_query)


def _gqa_dense_values(q, K, V, block_table, context_lens, scale, window, rows, num_query):
    """The decode oracle over pools of float64 values K, V [num_pages, P, Hkv, D], per (row,
    position, head): scores over the row's visible keys, max, exp, sum, weighted values."""
    if num_query == 1 and q.ndim == 3:
        q = q[:, None]
    B, Q, Hq, D = q.shape
    npg, P, Hkv, _ = K.shape
    G = Hq // Hkv
    qf = synth_bf16_to_f32(q).astype(np.float64)
    bt = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(context_lens, dtype=np.int64)
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(Q) for h in range(Hq)]
    elif len(rows) and len(rows[0]) == 2:
        rows = [(b, 0, h) for b, h in rows]
    o = np.zeros((len(rows), D))
    lse = np.full(len(rows), -np.inf)
    for n, (b, i, h) in enumerate(rows):
        hi = max(int(lens[b]) - Q + 1 + i, 0)
        lo = max(hi - window, 0) if window > 0 else 0
        if hi <= lo:
            continue
        t = np.arange(lo, hi)
        pages = bt[b, t // P]
        k = K[pages, t % P, h // G]
        v = V[pages, t % P, h // G]
        s = float(scale) * (k @ qf[b, i, h])
        m = s.max()
        p = np.exp(s - m)
        o[n] = (p / p.sum()) @ v
        lse[n] = m + np.log(p.sum())
    return o, lse


def synth_bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gqa_fp8(q, k_codes, v_codes, block_table, context_lens, scale: float, k_scale: float, v_scale: float,
            window: int = 0, rows=None, num_query: int = 1):
    """GQA decode (or multi-query verify with num_query > 1, q [B, Q, Hq, D]) over an FP8 cache,
    in float64: the attention of the decode oracle with keys decode(K code) * k_scale and values
    decode(V code) * v_scale.  Written out per (row, head) with numpy: scores over the row's
    visible keys, max, exp, sum, weighted values.  Returns (o [n, D], lse [n])."""
    q = np.asarray(q, dtype=np.uint16)
    if num_query == 1 and q.ndim == 3:
        q = q[:, None]
    B, Q, Hq, D = q.shape
    npg, P, Hkv, _ = k_codes.shape
    G = Hq // Hkv
    qf = synth_bf16_to_f32(q).astype(np.float64)
    K = e4m3_decode(k_codes) * float(np.float32(k_scale))
    V = e4m3_decode(v_codes) * float(np.float32(v_scale))
    bt = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(context_lens, dtype=np.int64)
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(Q) for h in range(Hq)]
    elif len(rows) and len(rows[0]) == 2:
        rows = [(b, 0, h) for b, h in rows]
    o = np.zeros((len(rows), D))
    lse = np.full(len(rows), -np.inf)
    for n, (b, i, h) in enumerate(rows):
        hi = max(int(lens[b]) - Q + 1 + i, 0)
        lo = max(hi - window, 0) if window > 0 else 0
        if hi <= lo:
            continue
        t = np.arange(lo, hi)
        pages = bt[b, t // P]
        k = K[pages, t % P, h // G]
        v = V[pages, t % P, h // G]
        s = float(scale) * (k @ qf[b, i, h])
        m = s.max()
        p = np.exp(s - m)
        o[n] = (p / p.sum()) @ v
        lse[n] = m + np.log(p.sum())
    return o, lse
