"""Seeded synthetic inputs for paged decode attention.

This module is the one piece shared by the CUDA path's tests/bench and the
fp64 oracle's tests.  It only *draws numbers and lays them out*: it holds none
of the attention arithmetic (no dot products, no softmax, no merge).

Recipe (all counter-based, so any element can be regenerated on its own):

* ``splitmix64``: output ``i`` of stream ``s`` is ``mix(s + (i + 1) * GOLDEN)``
  (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; the finaliser is the published variant-13 mixer).
* ``normal``: Box-Muller (cosine branch) on two consecutive outputs,
  ``u1 = (x >> 11 + 1) * 2^-53`` in (0, 1], ``u2 = (y >> 11) * 2^-53`` in [0, 1).
* bf16 values: float64 normal * std -> float32 (RNE) -> bf16 (RNE), stored as
  raw ``uint16`` bit patterns.  Both sides of every parity test consume exactly
  these bits.
* context lengths: uniform integers on an inclusive range, or log-uniform as
  ``floor(exp(U(ln a, ln b)))``, or a fixed list.
* page pool: holds ``sum_b ceil(L_b / P)`` pages times an oversize factor.  A
  seeded Fisher-Yates permutation assigns physical pages to logical pages.
  Every slot that the attention must not read (unused pool pages, the tail of
  each row's last page, pages wholly outside a sliding window) is filled with a
  bf16 NaN, so a stray read poisons the result.
* Data is drawn per *logical* (row, token, head, dim) coordinate, so the same
  seed gives the same logical cache under any physical page permutation.
* FP8 (E4M3) pools hold codes drawn directly (no conversion from values):
  output ``x`` of the element's stream gives the sign (bit 0) and, with
  probability 1/32 (bits 1-5 all zero), a 7-bit magnitude code uniform over all
  127 finite ones (zeros, subnormals, 448 included), else one uniform over
  0x28..0x6F (values 0.25 .. 120, log-uniform).  Slots that must not be read
  hold the NaN code 0x7F.
* NVFP4 pools hold row bytes drawn directly the same way.  A row of D values is
  D / 2 code bytes, D / 16 block-scale codes and zero padding to a multiple of
  16 bytes.  Output ``x`` of a code byte's stream gives the byte (``x & 255``:
  two uniform 4-bit codes).  A scale byte's ``x`` gives, with probability 1/32
  (bits 8-12 all zero), a code uniform over 0x00..0x4F (zero, the subnormals,
  normals up to 7.5), else one uniform over 0x28..0x47 (0.25 .. 3.75).  Slots
  that must not be read hold 0x7F in every byte (a NaN block scale).

The workloads mirror the decode shapes of the pages: the Llama-3-8B / Qwen3-32B
GQA geometries and the 576-wide (512 latent + 64 rope) MLA cache of
DeepSeek-V2-Lite named in the vllm.cpp kernel-matrix rows KERNEL-ATTN-FA2 and
KERNEL-ATTN-MLA-SPARSE.  No public dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)

# stream tags: one independent splitmix64 stream per drawn quantity
TAG_Q, TAG_K, TAG_V, TAG_LENS, TAG_PERM, TAG_CACHE, TAG_WUK, TAG_WUV, TAG_SLOT = range(1, 10)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(state: int, index: np.ndarray) -> np.ndarray:
    """Outputs ``index`` (0-based, uint64 array) of the splitmix64 stream seeded with ``state``."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(state) + (idx + np.uint64(1)) * GOLDEN)


def stream_seed(seed: int, tag: int) -> int:
    """Seed of the independent sub-stream ``tag`` of the workload seed ``seed``."""
    with np.errstate(over="ignore"):
        return int(splitmix64(seed, np.array([tag], dtype=np.uint64))[0])


def uniform01(state: int, index: np.ndarray) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of each stream output."""
    return (splitmix64(state, index) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(state: int, index: np.ndarray) -> np.ndarray:
    """Standard normal doubles, one per ``index``; uses stream outputs 2i and 2i+1."""
    idx = np.asarray(index, dtype=np.uint64)
    x = splitmix64(state, idx * np.uint64(2))
    y = splitmix64(state, idx * np.uint64(2) + np.uint64(1))
    u1 = ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (y >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); NaN stays a quiet NaN."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(state: int, index: np.ndarray, std: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits((normal(state, index) * std).astype(np.float32))


def _normal_bf16_range(state: int, start: int, n: int, std: float, chunk: int = 1 << 18) -> np.ndarray:
    """bf16 normals for stream indices [start, start + n), drawn in cache-sized chunks."""
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = normal_bf16(state, np.arange(start + s, start + e, dtype=np.uint64), std)
    return out


def _normal_bf16_dense(state: int, n: int, std: float) -> np.ndarray:
    return _normal_bf16_range(state, 0, n, std)


def e4m3_codes(state: int, index: np.ndarray) -> np.ndarray:
    """FP8 E4M3 codes (uint8), one per ``index``, by the recipe in the module docstring."""
    x = splitmix64(state, index)
    sign = (x & np.uint64(1)).astype(np.uint8) << np.uint8(7)
    wide = ((x >> np.uint64(1)) & np.uint64(31)) == 0
    r = x >> np.uint64(8)
    mag = np.where(wide, r % np.uint64(127), np.uint64(0x28) + r % np.uint64(0x48)).astype(np.uint8)
    return sign | mag


def _codes_range(state: int, start: int, n: int, chunk: int = 1 << 18) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = e4m3_codes(state, np.arange(start + s, start + e, dtype=np.uint64))
    return out


def nvfp4_row_bytes(head_dim: int) -> int:
    """Bytes of one NVFP4 row (layout only): head_dim / 2 code bytes, head_dim / 16 scale codes,
    zero padding to a multiple of 16."""
    return (head_dim // 2 + head_dim // 16 + 15) // 16 * 16


def nvfp4_bytes(state: int, index: np.ndarray, head_dim: int) -> np.ndarray:
    """NVFP4 row bytes (uint8), one per ``index`` (its place in a row is index % row bytes), by
    the recipe in the module docstring."""
    R = nvfp4_row_bytes(head_dim)
    o = (np.asarray(index, dtype=np.uint64) % np.uint64(R)).astype(np.int64)
    x = splitmix64(state, index)
    code = (x & np.uint64(255)).astype(np.uint8)
    wide = ((x >> np.uint64(8)) & np.uint64(31)) == 0
    r = x >> np.uint64(16)
    sc = np.where(wide, r % np.uint64(0x50), np.uint64(0x28) + r % np.uint64(0x20)).astype(np.uint8)
    return np.where(o < head_dim // 2, code, np.where(o < head_dim // 2 + head_dim // 16, sc, np.uint8(0)))


def _nvfp4_range(state: int, start: int, n: int, head_dim: int, chunk: int = 1 << 18) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = nvfp4_bytes(state, np.arange(start + s, start + e, dtype=np.uint64), head_dim)
    return out


def permutation(state: int, n: int) -> np.ndarray:
    """Seeded Fisher-Yates shuffle of range(n) (Durstenfeld form, j drawn from [0, i])."""
    perm = np.arange(n, dtype=np.int64)
    if n <= 1:
        return perm
    u = uniform01(state, np.arange(n, dtype=np.uint64))
    for i in range(n - 1, 0, -1):
        j = int(u[i] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


def context_lengths(seed: int, batch: int, dist: str, lo: int = 0, hi: int = 0,
                    values: Optional[Sequence[int]] = None) -> np.ndarray:
    """Per-row context lengths: ``fixed`` list, ``uniform`` on [lo, hi], or ``loguniform`` on [lo, hi]."""
    if dist == "fixed":
        assert values is not None and len(values) == batch
        return np.asarray(values, dtype=np.int32)
    u = uniform01(stream_seed(seed, TAG_LENS), np.arange(batch, dtype=np.uint64))
    if dist == "uniform":
        lens = lo + np.floor(u * (hi - lo + 1)).astype(np.int64)
    elif dist == "loguniform":
        lens = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
    else:
        raise ValueError(dist)
    return np.clip(lens, lo, hi).astype(np.int32)


def visible_range(L: int, window: int, num_query: int = 1) -> tuple:
    """Token range [lo, L) some query of a row attends to.  A row of length L holding Q new
    tokens has query positions i < Q at logical positions L - Q + i; position i attends to the
    keys up to and including its own, the W most recent of them when window W > 0.  The union
    over positions is [max(0, L - Q + 1 - W), L) (Q = 1: the W most recent keys)."""
    lo = max(0, L - num_query + 1 - window) if window > 0 else 0
    return lo, L


@dataclasses.dataclass
class PagedLayout:
    """Block table + pool geometry shared by the GQA and MLA workloads."""
    page_size: int
    context_lens: np.ndarray          # [B] int32
    block_table: np.ndarray           # [B, max_pages_per_seq] int32, -1 past the row's pages
    num_pages: int                    # physical pages in the pool
    logical_page_of_row: np.ndarray   # [B] first global logical page index of each row
    phys_of_logical: np.ndarray       # [total logical pages] physical page id

    @property
    def batch(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])


def make_layout(seed: int, context_lens: np.ndarray, page_size: int, pool_factor: int = 1,
                scramble: bool = True, extra_table_cols: int = 0) -> PagedLayout:
    lens = np.asarray(context_lens, dtype=np.int32)
    B = lens.shape[0]
    pages = [(int(L) + page_size - 1) // page_size for L in lens]
    total = int(sum(pages))
    num_pages = max(1, total * pool_factor)
    perm = permutation(stream_seed(seed, TAG_PERM), num_pages) if scramble else np.arange(num_pages)
    phys_of_logical = perm[:total].astype(np.int32)
    max_pages = max(1, max(pages) + extra_table_cols)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    first = np.zeros(B, dtype=np.int64)
    off = 0
    for b in range(B):
        first[b] = off
        table[b, : pages[b]] = phys_of_logical[off: off + pages[b]]
        off += pages[b]
    return PagedLayout(page_size, lens, table, num_pages, first, phys_of_logical)


def _fill_pool(state: int, layout: PagedLayout, row_width: int, std: float, window: int,
               visible_only: bool, num_query: int = 1, fp8: bool = False, nvfp4_dim: int = 0) -> np.ndarray:
    """Pool [num_pages, P, row_width] bf16 bits (fp8: E4M3 codes; nvfp4_dim > 0: NVFP4 row bytes of
    that head_dim); values drawn per logical (page, slot, element)."""
    P = layout.page_size
    byte_pool = fp8 or nvfp4_dim > 0
    poison = E4M3_NAN if byte_pool else BF16_NAN
    pool = np.full((layout.num_pages, P, row_width), poison, dtype=np.uint8 if byte_pool else np.uint16)
    per_page = P * row_width
    for b in range(layout.batch):
        L = int(layout.context_lens[b])
        if L == 0:
            continue
        lo, hi = visible_range(L, window, num_query) if visible_only else (0, L)
        p0, p1 = lo // P, (hi + P - 1) // P
        g0 = int(layout.logical_page_of_row[b])
        if nvfp4_dim > 0:
            vals = _nvfp4_range(state, (g0 + p0) * per_page, (p1 - p0) * per_page, nvfp4_dim)
        elif fp8:
            vals = _codes_range(state, (g0 + p0) * per_page, (p1 - p0) * per_page)
        else:
            vals = _normal_bf16_range(state, (g0 + p0) * per_page, (p1 - p0) * per_page, std)
        vals = vals.reshape(p1 - p0, P, row_width)
        flat = vals.reshape((p1 - p0) * P, row_width)
        # poison the slots of the visited pages that lie outside [lo, hi)
        flat[: lo - p0 * P] = poison
        flat[hi - p0 * P:] = poison
        pool[layout.block_table[b, p0:p1]] = vals
    return pool


@dataclasses.dataclass
class GQAWorkload:
    name: str
    seed: int
    q: np.ndarray            # [B, Hq, D] bf16 bits ([B, Q, Hq, D] when num_query > 1)
    k_pool: np.ndarray       # [num_pages, P, Hkv, D] bf16 bits (fp8: uint8 E4M3 codes; nvfp4: [.., Hkv, R] uint8 rows)
    v_pool: np.ndarray       # the same for the values
    layout: PagedLayout
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    window: int
    k_std: float = 1.0
    num_query: int = 1
    fp8: bool = False
    k_scale: float = 1.0     # fp8: key = E4M3(code) * k_scale (nvfp4: the pool scale)
    v_scale: float = 1.0     # fp8: value = E4M3(code) * v_scale
    nvfp4: bool = False

    @property
    def batch(self):
        return self.layout.batch

    def visible_tokens(self) -> int:
        r = [visible_range(int(L), self.window, self.num_query) for L in self.layout.context_lens]
        return int(sum(hi - lo for lo, hi in r))

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move: every visible K and V row of each kv head once, all of q, and
        the output (every query position of a row shares the one walk over its keys)."""
        # per row: 2 bytes per value (bf16), 1 (FP8), or 9 / 16 (NVFP4: half a byte per value and a
        # scale byte per 16 values; the row's padding to 16 bytes is not counted)
        row = self.head_dim * 9 // 16 if self.nvfp4 else self.head_dim * (1 if self.fp8 else 2)
        kv = self.visible_tokens() * self.num_kv_heads * row * 2
        qb = self.batch * self.num_query * self.num_q_heads * self.head_dim * 2
        ob = self.batch * self.num_query * self.num_q_heads * (self.head_dim * 2 + 4)
        return kv + qb + ob


def make_gqa(seed: int, context_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
             page_size: int, window: int = 0, k_std: float = 1.0, pool_factor: int = 1,
             scale: Optional[float] = None, scramble: bool = True, name: str = "gqa",
             visible_only: bool = True, extra_table_cols: int = 0, num_query: int = 1,
             fp8: bool = False, k_scale: float = 1.0 / 64, v_scale: float = 1.0 / 128,
             nvfp4: bool = False) -> GQAWorkload:
    """GQA decode / verify inputs; fp8: E4M3 code pools, nvfp4: NVFP4 row pools, either with the
    given per-pool scales (k_std does not apply to them)."""
    lens = np.asarray(context_lens, dtype=np.int32)
    layout = make_layout(seed, lens, page_size, pool_factor, scramble, extra_table_cols)
    B = lens.shape[0]
    Q = num_query
    q = _normal_bf16_dense(stream_seed(seed, TAG_Q), B * Q * num_q_heads * head_dim, 1.0)
    q = q.reshape(B, num_q_heads, head_dim) if Q == 1 else q.reshape(B, Q, num_q_heads, head_dim)
    row = nvfp4_row_bytes(head_dim) if nvfp4 else head_dim
    w = num_kv_heads * row
    nd = head_dim if nvfp4 else 0
    k = _fill_pool(stream_seed(seed, TAG_K), layout, w, k_std, window, visible_only, Q, fp8, nd)
    v = _fill_pool(stream_seed(seed, TAG_V), layout, w, 1.0, window, visible_only, Q, fp8, nd)
    k = k.reshape(layout.num_pages, page_size, num_kv_heads, row)
    v = v.reshape(layout.num_pages, page_size, num_kv_heads, row)
    scaled = fp8 or nvfp4
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return GQAWorkload(name, seed, q, k, v, layout, num_q_heads, num_kv_heads, head_dim,
                       float(scale), int(window), float(k_std), int(Q), bool(fp8),
                       float(np.float32(k_scale)) if scaled else 1.0, float(np.float32(v_scale)) if scaled else 1.0,
                       bool(nvfp4))


MLA_NOPE, MLA_ROPE, MLA_LATENT, MLA_VDIM = 128, 64, 512, 128
MLA_QDIM = MLA_NOPE + MLA_ROPE          # 192
MLA_CDIM = MLA_LATENT + MLA_ROPE        # 576


@dataclasses.dataclass
class MLAWorkload:
    name: str
    seed: int
    q: np.ndarray       # [B, H, 192] bf16 bits: q_nope (128) || q_rope (64)
    cache: np.ndarray   # [num_pages, P, 576] bf16 bits: latent (512) || rope key (64)
    w_uk: np.ndarray    # [H, 128, 512] bf16 bits, W_UK[h][d][j]
    w_uv: np.ndarray    # [H, 128, 512] bf16 bits, W_UV[h][dv][j]
    layout: PagedLayout
    num_heads: int
    scale: float

    @property
    def batch(self):
        return self.layout.batch

    def visible_tokens(self) -> int:
        return int(sum(int(L) for L in self.layout.context_lens))

    def algorithmic_bytes(self, with_weights: bool = True) -> int:
        c = self.visible_tokens() * MLA_CDIM * 2
        qb = self.batch * self.num_heads * MLA_QDIM * 2
        ob = self.batch * self.num_heads * (MLA_VDIM * 2 + 4)
        wb = 2 * self.num_heads * MLA_NOPE * MLA_LATENT * 2 if with_weights else 0
        return c + qb + ob + wb


def make_mla(seed: int, context_lens, num_heads: int, page_size: int, w_std: float = 0.02,
             scale: Optional[float] = None, scramble: bool = True, pool_factor: int = 1,
             name: str = "mla") -> MLAWorkload:
    lens = np.asarray(context_lens, dtype=np.int32)
    layout = make_layout(seed, lens, page_size, pool_factor, scramble)
    B = lens.shape[0]
    q = _normal_bf16_dense(stream_seed(seed, TAG_Q), B * num_heads * MLA_QDIM, 1.0)
    q = q.reshape(B, num_heads, MLA_QDIM)
    cache = _fill_pool(stream_seed(seed, TAG_CACHE), layout, MLA_CDIM, 1.0, 0, True)
    n_w = num_heads * MLA_NOPE * MLA_LATENT
    w_uk = _normal_bf16_dense(stream_seed(seed, TAG_WUK), n_w, w_std).reshape(num_heads, MLA_NOPE, MLA_LATENT)
    w_uv = _normal_bf16_dense(stream_seed(seed, TAG_WUV), n_w, w_std).reshape(num_heads, MLA_VDIM, MLA_LATENT)
    if scale is None:
        scale = 1.0 / math.sqrt(MLA_QDIM)
    return MLAWorkload(name, seed, q, cache, w_uk, w_uv, layout, num_heads, float(scale))


# ---------------------------------------------------------------------------
# The named workloads (seed = 20260 + index in WORKLOADS).  Shapes follow the
# decode geometries the pages discuss.
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class KVWriteWorkload:
    """New tokens' K and V (or MLA latent + rope key) and their cache slots.

    Slots follow a prefill: token t is position t % page_size of page
    perm[t // page_size], the pages of a seeded permutation of the pool; every
    ``pad_every``-th token (if > 0) is a padding token with slot -1.  The pool
    starts as bf16 NaN everywhere, so a write to a wrong slot shows."""
    name: str
    seed: int
    k: np.ndarray         # [T, Hkv, D] uint16 bf16 bits (MLA: c_lat [T, 512])
    v: np.ndarray         # [T, Hkv, D] uint16 (MLA: k_rope [T, 64])
    slots: np.ndarray     # [T] int64
    num_pages: int
    page_size: int
    mla: bool = False
    fp8: bool = False          # quantizing write into E4M3 pools
    k_scale: float = 1.0
    v_scale: float = 1.0
    nvfp4: bool = False        # quantizing write into NVFP4 row pools

    @property
    def num_tokens(self) -> int:
        return int(self.slots.shape[0])

    def pool_shape(self):
        if self.mla:
            return (self.num_pages, self.page_size, 576)
        if self.nvfp4:
            return (self.num_pages, self.page_size, self.k.shape[1], nvfp4_row_bytes(self.k.shape[2]))
        return (self.num_pages, self.page_size) + tuple(self.k.shape[1:])

    def empty_pool(self) -> np.ndarray:
        if self.fp8 or self.nvfp4:
            return np.full(self.pool_shape(), E4M3_NAN, dtype=np.uint8)
        return np.full(self.pool_shape(), BF16_NAN, dtype=np.uint16)

    def algorithmic_bytes(self) -> int:
        """Bytes read (the bf16 new rows of the written tokens) plus bytes written (the same rows
        in the pools: one byte per value for FP8 pools, whole rows with their padding for NVFP4
        pools)."""
        written = int((self.slots >= 0).sum())
        row_in = (576 * 2) if self.mla else 2 * int(np.prod(self.k.shape[1:])) * 2
        if self.nvfp4:
            row_out = 2 * self.k.shape[1] * nvfp4_row_bytes(self.k.shape[2])
        else:
            row_out = row_in // 2 if self.fp8 else row_in
        return written * (row_in + row_out)


def make_kv_write(seed: int, num_tokens: int, num_kv_heads: int, head_dim: int, page_size: int,
                  num_pages: int, pad_every: int = 0, mla: bool = False, name: str = "kv-write") -> KVWriteWorkload:
    assert num_tokens <= num_pages * page_size
    perm = permutation(stream_seed(seed, TAG_PERM), num_pages)
    t = np.arange(num_tokens, dtype=np.int64)
    slots = perm[t // page_size] * page_size + t % page_size
    if pad_every > 0:
        slots[pad_every - 1::pad_every] = -1
    if mla:
        k = _normal_bf16_dense(stream_seed(seed, TAG_CACHE), num_tokens * 512, 1.0).reshape(num_tokens, 512)
        v = _normal_bf16_dense(stream_seed(seed, TAG_K), num_tokens * 64, 1.0).reshape(num_tokens, 64)
    else:
        n = num_tokens * num_kv_heads * head_dim
        k = _normal_bf16_dense(stream_seed(seed, TAG_K), n, 1.0).reshape(num_tokens, num_kv_heads, head_dim)
        v = _normal_bf16_dense(stream_seed(seed, TAG_V), n, 1.0).reshape(num_tokens, num_kv_heads, head_dim)
    return KVWriteWorkload(name, seed, k, v, slots.astype(np.int64), num_pages, page_size, mla)


WORKLOADS = ("tiny", "llama3-8b", "qwen3-32b", "hd256-window", "mla", "kv-write", "qwen3-32b-verify4",
             "qwen3-32b-fp8", "kv-write-fp8", "qwen3-32b-nvfp4", "kv-write-nvfp4")


def workload(name: str, seed: Optional[int] = None, scramble: bool = True):
    i = WORKLOADS.index(name)
    seed = 20260 + i if seed is None else seed
    if name == "tiny":
        lens = context_lengths(seed, 6, "fixed", values=[1, 31, 32, 33, 64, 100])
        return make_gqa(seed, lens, 8, 2, 128, 32, name=name, scramble=scramble)
    if name == "llama3-8b":
        lens = context_lengths(seed, 8, "uniform", 512, 4096)
        return make_gqa(seed, lens, 32, 8, 128, 16, k_std=0.5, pool_factor=2, name=name,
                        scramble=scramble)
    if name == "qwen3-32b":
        lens = context_lengths(seed, 32, "loguniform", 128, 16384)
        return make_gqa(seed, lens, 64, 8, 128, 32, name=name, scramble=scramble)
    if name == "hd256-window":
        lens = context_lengths(seed, 16, "uniform", 2048, 32768)
        return make_gqa(seed, lens, 16, 4, 256, 32, window=4096, name=name, scramble=scramble)
    if name == "mla":
        lens = context_lengths(seed, 16, "uniform", 1024, 8192)
        return make_mla(seed, lens, 128, 64, name=name, scramble=scramble)
    if name == "qwen3-32b-verify4":
        # speculative verify: the qwen3-32b rows (same lengths) with 4 query positions each
        lens = context_lengths(20262 if seed == 20266 else seed, 32, "loguniform", 128, 16384)
        return make_gqa(seed, lens, 64, 8, 128, 32, name=name, scramble=scramble, num_query=4)
    if name == "qwen3-32b-fp8":
        # the qwen3-32b rows (same lengths) over an FP8 E4M3 cache
        lens = context_lengths(20262 if seed == 20267 else seed, 32, "loguniform", 128, 16384)
        return make_gqa(seed, lens, 64, 8, 128, 32, name=name, scramble=scramble, fp8=True)
    if name == "kv-write-fp8":
        # the kv-write prefill chunk quantized into E4M3 pools (scales 1/64, 1/128)
        w = make_kv_write(20265 if seed == 20268 else seed, 16384, 8, 128, 32, 1024, name=name)
        return dataclasses.replace(w, fp8=True, k_scale=float(np.float32(1 / 64)), v_scale=float(np.float32(1 / 128)))
    if name == "qwen3-32b-nvfp4":
        # the qwen3-32b rows (same lengths) over an NVFP4 cache (pool scales 1/4 and 1/16)
        lens = context_lengths(20262 if seed == 20269 else seed, 32, "loguniform", 128, 16384)
        return make_gqa(seed, lens, 64, 8, 128, 32, name=name, scramble=scramble, nvfp4=True, k_scale=0.25,
                        v_scale=1.0 / 16)
    if name == "kv-write-nvfp4":
        # the kv-write prefill chunk quantized into NVFP4 pools (pool scales 1/4, 1/2)
        w = make_kv_write(20265 if seed == 20270 else seed, 16384, 8, 128, 32, 1024, name=name)
        return dataclasses.replace(w, nvfp4=True, k_scale=0.25, v_scale=0.5)
    if name == "kv-write":
        # a 16384-token prefill chunk into a Qwen3-32B-shaped cache (8 KV heads, D 128, page 32)
        return make_kv_write(seed, 16384, 8, 128, 32, 1024, name=name)
    raise KeyError(name)
