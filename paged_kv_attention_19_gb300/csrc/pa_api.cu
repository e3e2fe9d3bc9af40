// pa_api.cu -- the C ABI (include/pa_decode.h): argument validation, workspace
// layout, TMA tensor-map encoding and the launch sequence of each call.
//
// Every check that can be made on the host is made before anything is
// launched, so an invalid call returns an error code with no device work and
// no CUDA call at all.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_decode.h"
#include "pa_gqa.cuh"
#include "pa_launch.h"
#include "pa_mla.h"

namespace {

using namespace pa;

constexpr int kMaxSplits = 4096;     // largest accepted explicit num_splits (partitions)
constexpr int kAutoPartsMax = 256;   // automatic mode: one partition per SM, at most this many
constexpr int kMaxQueryPositions = 64;  // verify: query positions per row
// Fixed cost of one piece of work in the GQA partition, expressed as the KV bytes an SM
// streams meanwhile: the query load, the end-of-piece merge and the partial's share of the
// combine, and the start-up and tail of a piece's stages.  Set by measurement (sweeps of the
// qwen3-32b, hd256-window and llama3-8b decodes, and of the 4-position verify): a sequence of
// one 16-row tile...
constexpr long long kPieceCostBytes = 80 << 10;
// ...and one of two paired tiles, whose pieces copy both tiles' query rows and merge twice.
constexpr long long kPieceCostBytesPair = 192 << 10;
// The same for FP8 pools, whose pieces cost more (the query split and a merge over twice
// the token groups) while each byte carries twice the tokens.
constexpr long long kPieceCostBytesF8 = 128 << 10;
// NVFP4 pools: a byte carries about 3.2 times the tokens of bf16 (head_dim 128: 80-byte rows), so
// a piece's fixed cost is fewer bytes.  Swept on the NVFP4 qwen3-32b decode: 16 KB 61.9 us, 32 KB
// 59.3, 64 KB 61.2, 96 KB 65.2.
constexpr long long kPieceCostBytesFp4 = 32 << 10;

thread_local cudaEvent_t t_ev_before = nullptr;
thread_local cudaEvent_t t_ev_after = nullptr;
thread_local int t_last_launches = 0;
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
thread_local unsigned long long t_wait_limit_ns = WAIT_LIMIT_NS;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Element formats of the K/V pools.
enum PoolFmt { FMT_BF16 = 0, FMT_FP8 = 1, FMT_NVFP4 = 2 };

// Tokens per stage of the split kernel (must match GqaCfg<D>::ST, GqaF8Cfg<D, *>::ST and
// GqaFp4Cfg<D>::ST).
int gqa_stage_tokens(int D, int fmt) {
  if (fmt == FMT_FP8) return D <= 128 ? 128 : 64;
  if (fmt == FMT_NVFP4) return D <= 128 ? 128 : 32;
  return D <= 128 ? 64 : 32;
}

// Bytes of an NVFP4 pool row of D values (must match nvfp4_row_bytes in pa_gqa_fp4.cuh): D / 2
// bytes of code pairs, D / 16 block scales, zero padding to a multiple of 16 bytes.
int nvfp4_row(int D) { return (D / 2 + D / 16 + 15) / 16 * 16; }

struct GqaPlan {
  int nsub, nparts_max;
  size_t off_desc, off_part_lse, off_part_o, off_seq, total;
};

// Shape checks shared by pa_workspace_size and pa_decode_gqa; PA_OK or an error code.
// The workspace holds the header, one descriptor per partition, two fp32 partial
// slots (32 rows -- two 16-row tiles -- x head_dim, plus their LSEs) per
// partition, and two int32 tables of where each sequence's pieces are: one
// entry each per (row, KV head, tile) for the largest query count a call may
// have (kMaxQueryPositions).  Its size does not depend on the context lengths.
int gqa_shape(int batch, int Hq, int Hkv, int D, int max_ctx, int P, int num_splits, GqaPlan *pl) {
  if (batch < 0 || Hq <= 0 || Hkv <= 0 || max_ctx < 0 || num_splits < 0) return PA_ERR_INVALID_ARGUMENT;
  if (Hq % Hkv != 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_splits > kMaxSplits) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(P) || P < 8 || P > 256) return PA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  pl->nsub = (G + 15) / 16;  // query heads per tensor-core tile: 16
  pl->nparts_max = num_splits > 0 ? num_splits : kAutoPartsMax;
  const size_t np = (size_t)pl->nparts_max;
  size_t off = sizeof(WsHeader);
  pl->off_desc = off;
  off = round_up(off + np * sizeof(GqaPartDesc), 256);
  pl->off_part_lse = off;
  off = round_up(off + np * 2 * PART_ROWS * sizeof(float), 256);
  pl->off_part_o = off;
  off = round_up(off + np * 2 * PART_ROWS * (size_t)D * sizeof(float), 256);
  pl->off_seq = off;
  const size_t max_seqs = (size_t)(batch > 0 ? batch : 1) * Hkv * kMaxQueryPositions * pl->nsub;
  off = round_up(off + 2 * max_seqs * sizeof(int32_t), 256);
  pl->total = off;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D map over a [num_pages, P, H, D] pool of bf16 (esz 2) or FP8 (esz 1) values; box = (one
// 128-byte row fragment: 64 or 128 dims, 1 head, BH tokens, 1 page), written to shared memory
// with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap *m, const void *base, int num_pages, int P, int H, int D, int BH, int esz = 2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t e = (cuuint64_t)esz;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)P, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)D * e, (cuuint64_t)H * D * e, (cuuint64_t)P * H * D * e};
  cuuint32_t box[4] = {128u / (cuuint32_t)esz, 1u, (cuuint32_t)BH, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = fn(m, esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D map over a [num_pages, P, H, D] pool of bf16 values seen as (64 dims, P tokens, D / 64
// planes, H heads, pages): the plane stride (128 bytes) is below the token stride.  Box = (64 dims,
// BH tokens, all planes, 1 head, 1 page): one copy brings a unit's rows of every plane, landing as
// the planes' BH 128-byte rows one after the other, with the 128-byte swizzle (the unit-major stage
// blocks of the bf16 split kernel, head_dim 128 and 256).
bool encode_pool_units_map(CUtensorMap *m, const void *base, int num_pages, int P, int H, int D, int BH) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[5] = {64u, (cuuint64_t)P, (cuuint64_t)(D / 64), (cuuint64_t)H, (cuuint64_t)num_pages};
  cuuint64_t strides[4] = {(cuuint64_t)H * D * 2, 128u, (cuuint64_t)D * 2, (cuuint64_t)P * H * D * 2};
  cuuint32_t box[5] = {64u, (cuuint32_t)BH, (cuuint32_t)(D / 64), 1u, 1u};
  cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D map over a [num_pages, P, H, R] pool of NVFP4 rows (R bytes each); box = (one whole row,
// 1 head, BH tokens, 1 page), no swizzle: the box's rows land as consecutive R-byte rows.
bool encode_nvfp4_map(CUtensorMap *m, const void *base, int num_pages, int P, int H, int R, int BH) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)P, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)R, (cuuint64_t)H * R, (cuuint64_t)P * H * R};
  cuuint32_t box[4] = {(cuuint32_t)R, 1u, (cuuint32_t)BH, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over q viewed as [batch * Q positions, Hq, D] bf16; box = (64 dims, gt heads, qt
// positions), 128-byte swizzle: the qt x gt rows of one tile land as consecutive 128-byte rows.
bool encode_q_map(CUtensorMap *m, const void *base, long long positions, int Hq, int D, int gt, int qt) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)positions};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)gt, (cuuint32_t)qt};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= 64) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}


}  // namespace

namespace pa {
void note_launches(int n) { t_last_launches = n; }
int cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  t_last_cuda_error = e == cudaSuccess ? cudaErrorUnknown : e;
  return PA_ERR_CUDA;
}
cudaError_t profile_mark(bool before, cudaStream_t stream) {
  cudaEvent_t e = before ? t_ev_before : t_ev_after;
  return e ? cudaEventRecord(e, stream) : cudaSuccess;
}
}  // namespace pa

extern "C" {

size_t pa_workspace_size(int kind, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_context_len, int page_size, int num_splits) {
  if (kind == PA_KIND_GQA) {
    GqaPlan pl;
    if (gqa_shape(batch, num_q_heads, num_kv_heads, head_dim, max_context_len, page_size, num_splits, &pl) !=
        PA_OK)
      return 0;
    return pl.total;
  }
  if (kind == PA_KIND_MLA_ABSORBED) {
    return pa::mla_workspace_size(batch, num_q_heads, max_context_len, page_size, num_splits);
  }
  return 0;
}

}  // extern "C"

namespace {

// Pool format and scales: one float per pool (FP8 and NVFP4), each finite and positive.
struct PoolScales {
  int fmt;
  float k, v;
};

// GQA decode (Q == 1) and verify (Q > 1 query positions per row, causal among them), over
// bf16 pools, FP8 E4M3 pools or NVFP4 pools, the last two with per-pool scales.
int gqa_call(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
             const int32_t *context_lens, void *out, float *lse, int batch, int Q, int num_q_heads,
             int num_kv_heads, int head_dim, int page_size, int num_pages, int max_pages_per_seq,
             int max_context_len, float scale, int window, int num_splits, void *workspace,
             size_t workspace_bytes, cudaStream_t stream, PoolScales f8 = {FMT_BF16, 1.f, 1.f}) {
  t_last_launches = 0;
  const bool fp8 = f8.fmt == FMT_FP8, fp4 = f8.fmt == FMT_NVFP4, scaled = fp8 || fp4;
  if (Q <= 0 || Q > kMaxQueryPositions) return Q <= 0 ? PA_ERR_INVALID_ARGUMENT : PA_ERR_UNSUPPORTED;
  if (scaled && !(std::isfinite(f8.k) && f8.k > 0.f && std::isfinite(f8.v) && f8.v > 0.f))
    return PA_ERR_INVALID_ARGUMENT;
  if (batch == 0) return PA_OK;
  GqaPlan pl;
  int rc = gqa_shape(batch, num_q_heads, num_kv_heads, head_dim, max_context_len, page_size, num_splits, &pl);
  if (rc != PA_OK) return rc;
  if (fp8 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (!q || !k_pool || !v_pool || !block_table || !context_lens || !out || !workspace)
    return PA_ERR_INVALID_ARGUMENT;
  if (num_pages <= 0 || max_pages_per_seq <= 0 || !std::isfinite(scale)) return PA_ERR_INVALID_ARGUMENT;
  if ((long long)max_pages_per_seq * page_size < (long long)max_context_len) return PA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16) || !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      (lse && !aligned(lse, 4)))
    return PA_ERR_MISALIGNED;
  if (workspace_bytes < pl.total) return PA_ERR_WORKSPACE_TOO_SMALL;

  const int D = head_dim, P = page_size;
  const int ST = gqa_stage_tokens(D, f8.fmt);
  const int BH = P < ST ? P : ST;  // tokens per TMA box = per work unit
  // query tiles of at most 16 MMA rows: qt positions x gt heads of one KV head's group
  const int G = num_q_heads / num_kv_heads;
  const int gt = G < PART_HEADS ? G : PART_HEADS;
  const int qt = G < PART_HEADS ? (Q < PART_HEADS / G ? Q : PART_HEADS / G) : 1;
  const int ntile = G < PART_HEADS ? (Q + qt - 1) / qt : Q * pl.nsub;
  // a KV head with more than one tile has its tiles paired in one sequence (bf16 pools, head_dim
  // up to 128: both tiles' fragments fit the consumers' registers), so a page crosses shared
  // memory once for all of the head's rows
  const int mt = (!scaled && D <= 128 && ntile >= 2) ? 2 : 1;
  const int nseqh = (ntile + mt - 1) / mt;
  CUtensorMap tm_k, tm_v, tm_q;
  const int esz = fp8 ? 1 : 2;
  // decode over bf16 pages of fewer than 32 tokens with more than one 64-dim plane: the unit-major
  // kernel, whose producer fills a unit of all planes by one 5-D copy
  const bool units = !fp8 && !fp4 && D > 64 && BH < 32 && Q == 1 && mt == 1;
  const bool maps_ok =
      fp4     ? encode_nvfp4_map(&tm_k, k_pool, num_pages, P, num_kv_heads, nvfp4_row(D), BH) &&
                encode_nvfp4_map(&tm_v, v_pool, num_pages, P, num_kv_heads, nvfp4_row(D), BH)
      : units ? encode_pool_units_map(&tm_k, k_pool, num_pages, P, num_kv_heads, D, BH) &&
                encode_pool_units_map(&tm_v, v_pool, num_pages, P, num_kv_heads, D, BH)
              : encode_pool_map(&tm_k, k_pool, num_pages, P, num_kv_heads, D, BH, esz) &&
                encode_pool_map(&tm_v, v_pool, num_pages, P, num_kv_heads, D, BH, esz);
  if (!maps_ok || !encode_q_map(&tm_q, q, (long long)batch * Q, num_q_heads, D, gt, qt)) return PA_ERR_UNSUPPORTED;
  const int sms = sm_count();
  if (sms <= 0) return pa::cuda_fail(cudaSuccess);
  const int nparts = num_splits > 0 ? num_splits : (sms < kAutoPartsMax ? sms : kAutoPartsMax);

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  GqaPartDesc *desc = reinterpret_cast<GqaPartDesc *>(ws + pl.off_desc);
  float *part_lse = reinterpret_cast<float *>(ws + pl.off_part_lse);
  float *part_o = reinterpret_cast<float *>(ws + pl.off_part_o);
  const int hs = num_kv_heads * nseqh;  // sequences per row
  int32_t *seq_first = reinterpret_cast<int32_t *>(ws + pl.off_seq);
  int32_t *seq_last = seq_first + (size_t)batch * hs;

  GqaArgs ga;
  ga.q = static_cast<const uint16_t *>(q);
  ga.block_table = block_table;
  ga.context_lens = context_lens;
  ga.out = static_cast<uint16_t *>(out);
  ga.lse = lse;
  ga.part_o = part_o;
  ga.part_lse = part_lse;
  ga.desc = desc;
  ga.seq_first = seq_first;
  ga.seq_last = seq_last;
  ga.batch = batch;
  ga.max_pages_per_seq = max_pages_per_seq;
  ga.num_pages = num_pages;
  ga.max_context_len = max_context_len;
  ga.window = window > 0 ? window : 0;
  ga.Hq = num_q_heads;
  ga.Hkv = num_kv_heads;
  ga.G = num_q_heads / num_kv_heads;
  ga.nsub = pl.nsub;
  ga.Q = Q;
  ga.gt = gt;
  ga.qt = qt;
  ga.ntile = ntile;
  ga.mt = mt;
  ga.nseqh = nseqh;
  ga.log2_page = ilog2(P);
  ga.log2_bh = ilog2(BH);
  ga.unit_copy = units ? 1 : 0;
  ga.nparts = nparts;
  ga.hg = hs < nparts ? hs : nparts;
  {
    // K and V of one unit of one KV head
    const long long unit_bytes = (long long)BH * 2 * (fp4 ? nvfp4_row(D) : D * esz);
    const long long piece_bytes = fp8 ? kPieceCostBytesF8
                                  : fp4 ? kPieceCostBytesFp4
                                        : mt == 2 ? kPieceCostBytesPair : kPieceCostBytes;
    ga.piece_cost = (int)((piece_bytes + unit_bytes - 1) / unit_bytes);
  }
  ga.qscale = scale * LOG2E * (scaled ? f8.k : 1.f);
  ga.vscale = scaled ? f8.v : 1.f;
  ga.wait_ns = t_wait_limit_ns;

  CombineArgs ca;
  ca.out = static_cast<uint16_t *>(out);
  ca.lse = lse;
  ca.part_o = part_o;
  ca.part_lse = part_lse;
  ca.desc = desc;
  ca.seq_first = seq_first;
  ca.seq_last = seq_last;
  ca.context_lens = context_lens;
  ca.status = &hdr->status;
  ca.Hq = num_q_heads;
  ca.G = ga.G;
  ca.nsub = pl.nsub;
  ca.nparts = nparts;
  ca.hg = ga.hg;
  ca.Q = Q;
  ca.gt = gt;
  ca.qt = qt;
  ca.ntile = ntile;
  ca.mt = mt;
  ca.nseqh = nseqh;
  ca.hs = hs;
  ca.max_context_len = max_context_len;
  ca.nblocks = batch * hs;

  cudaError_t e;
  if (t_ev_before) {
    if (const cudaError_t ce = cudaEventRecord(t_ev_before, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  }
  if (fp4) {
    e = launch_gqa_split_nvfp4(D, nparts, tm_k, tm_v, tm_q, ga, stream);
  } else if (fp8) {
    e = D == 128 ? launch_gqa_split_fp8_d128(nparts, tm_k, tm_v, tm_q, ga, stream)
                 : launch_gqa_split_fp8_d256(nparts, tm_k, tm_v, tm_q, ga, stream);
  } else {
    switch (D) {
      case 64: e = launch_gqa_split_d64(nparts, tm_k, tm_v, tm_q, ga, stream); break;
      case 128: e = launch_gqa_split_d128(nparts, tm_k, tm_v, tm_q, ga, stream); break;
      default: e = launch_gqa_split_d256(nparts, tm_k, tm_v, tm_q, ga, stream); break;
    }
  }
  if (e != cudaSuccess) return pa::cuda_fail(e);
  ++t_last_launches;
  if (t_ev_after) {
    if (const cudaError_t ce = cudaEventRecord(t_ev_after, stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  }
  switch (D) {
    case 64: e = launch_gqa_combine_d64(ca, stream); break;
    case 128: e = launch_gqa_combine_d128(ca, stream); break;
    default: e = launch_gqa_combine_d256(ca, stream); break;
  }
  if (e != cudaSuccess) return pa::cuda_fail(e);
  ++t_last_launches;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode_gqa(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
                  const int32_t *context_lens, void *out, float *lse, int batch, int num_q_heads,
                  int num_kv_heads, int head_dim, int page_size, int num_pages, int max_pages_per_seq,
                  int max_context_len, float scale, int window, int num_splits, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
  return gqa_call(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, 1, num_q_heads, num_kv_heads,
                  head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window, num_splits,
                  workspace, workspace_bytes, stream);
}

int pa_verify_gqa(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
                  const int32_t *context_lens, void *out, float *lse, int batch, int num_query,
                  int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                  int max_pages_per_seq, int max_context_len, float scale, int window, int num_splits,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  return gqa_call(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, num_query, num_q_heads,
                  num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window,
                  num_splits, workspace, workspace_bytes, stream);
}

int pa_decode_gqa_fp8(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
                      const int32_t *context_lens, void *out, float *lse, int batch, int num_query,
                      int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                      int max_pages_per_seq, int max_context_len, float scale, float k_scale, float v_scale,
                      int window, int num_splits, void *workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  return gqa_call(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, num_query, num_q_heads,
                  num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window,
                  num_splits, workspace, workspace_bytes, stream, PoolScales{FMT_FP8, k_scale, v_scale});
}

int pa_decode_gqa_nvfp4(const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
                        const int32_t *context_lens, void *out, float *lse, int batch, int num_query,
                        int num_q_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                        int max_pages_per_seq, int max_context_len, float scale, float k_scale, float v_scale,
                        int window, int num_splits, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  return gqa_call(q, k_pool, v_pool, block_table, context_lens, out, lse, batch, num_query, num_q_heads,
                  num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq, max_context_len, scale, window,
                  num_splits, workspace, workspace_bytes, stream, PoolScales{FMT_NVFP4, k_scale, v_scale});
}

int pa_decode_mla_absorbed(const void *q, const void *cache, const void *w_uk, const void *w_uv,
                           const int32_t *block_table, const int32_t *context_lens, void *out, float *lse,
                           int batch, int num_heads, int page_size, int num_pages, int max_pages_per_seq,
                           int max_context_len, float scale, int num_splits, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  t_last_launches = 0;
  int launches = 0;
  const int rc = pa::mla_decode(q, cache, w_uk, w_uv, block_table, context_lens, out, lse, batch, num_heads,
                                page_size, num_pages, max_pages_per_seq, max_context_len, scale, num_splits,
                                workspace, workspace_bytes, stream, t_ev_before, t_ev_after, &launches);
  t_last_launches = launches;
  return rc;
}

const char *pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case PA_ERR_MISALIGNED: return "misaligned pointer";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int pa_read_device_status(const void *workspace, cudaStream_t stream, uint32_t *out_bits) {
  if (!workspace || !out_bits) return PA_ERR_INVALID_ARGUMENT;
  if (!aligned(workspace, 16)) return PA_ERR_MISALIGNED;
  uint32_t v = 0;
  if (const cudaError_t ce = cudaStreamSynchronize(stream); ce != cudaSuccess) return pa::cuda_fail(ce);
  if (const cudaError_t ce = cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost); ce != cudaSuccess) return pa::cuda_fail(ce);
  *out_bits = v;
  return PA_OK;
}

int pa_set_profile_events(cudaEvent_t before_main, cudaEvent_t after_main) {
  if ((before_main == nullptr) != (after_main == nullptr)) return PA_ERR_INVALID_ARGUMENT;
  t_ev_before = before_main;
  t_ev_after = after_main;
  return PA_OK;
}

int pa_last_launch_count(void) { return t_last_launches; }

int pa_set_wait_limit_ns(unsigned long long limit_ns) {
  t_wait_limit_ns = limit_ns;
  return PA_OK;
}

int pa_last_cuda_error(void) { return (int)t_last_cuda_error; }

const char *pa_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

}  // extern "C"
