/*
 * pa_decode.h -- C ABI of the paged decode attention library (GB300, sm_103a).
 *
 * Single-token decode (and speculative-verify) attention of a batch of query
 * rows against a paged KV cache, and the write of new tokens into the cache:
 *
 *   pa_decode_gqa           grouped-query attention, optional sliding window
 *   pa_verify_gqa           the same for several query positions per row
 *   pa_decode_gqa_fp8       both over an FP8 (E4M3) cache with per-pool scales
 *   pa_decode_gqa_nvfp4     both over an NVFP4 cache (E2M1 values, E4M3 block scales)
 *   pa_decode_mla_absorbed  multi-head latent attention in the absorbed form
 *   pa_kv_write, pa_kv_write_fp8, pa_kv_write_nvfp4, pa_mla_cache_write
 *                           the paged writes
 *
 * The operations are the ones the following pages describe:
 *   - paged cache: K/V pools [pages, block_size, Hkv, D], per-request
 *     seq_lens, and a block table (vllm.cpp kernel-matrix, rows
 *     KERNEL-ATTN-PAGED and KERNEL-ATTN-DFLASH-PAGED-BLOCK);
 *   - query heads sharing one KV head, served by one CTA per (batch, KV head)
 *     so that every KV page is read once per group (vllm.cpp PR #49 "flip
 *     decode GQA group-swap default ON", mechanism paragraph);
 *   - f32 online softmax over the KV sequence and the HasWindow arm
 *     (vllm.cpp PR #425 "head_dim-128 arm for the warp-split-KV decode
 *     kernel", description and limitations list);
 *   - split-KV over the sequence with a separate combine step that merges
 *     splits in a fixed ascending order, no atomics on the data, empty splits
 *     skipped (kernel-matrix rows KERNEL-ATTN-FA2 and KERNEL-ATTN-MLA-SPARSE;
 *     for MLA the combine runs inside the W_UV projection's launch);
 *   - the absorbed MLA schedule q_lat = q_nope.W_UK || q_rope, scores over
 *     the 576-wide latent cache, o_lat = sum p c, o = W_UV.o_lat (pegainfer
 *     PR #938 "warp-cooperative two-pass MLA absorbed decode kernel",
 *     Schedule section, steps 1-7; kernel-matrix row KERNEL-ATTN-MLA-SPARSE,
 *     weight absorption as two batched contractions);
 *   - the paged writes and the FP8 and NVFP4 forms of the cache (kernel-matrix
 *     rows KERNEL-KV-CACHE and KERNEL-KV-QUANT);
 *   - the raw pointer / shape / scalar / workspace / stream calling
 *     convention of the planned drop-in kernel ABI (kernel-matrix preamble).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is DEVICE memory owned by the caller; the library
 *     allocates nothing at call time and keeps no state between calls
 *     (re-entrant).  The only library state is per host thread (the optional
 *     profiling hook, the launch count, the last CUDA error) and the fixed
 *     scratch array of pa_decode_gqa_noalloc.
 *   - Tensors are dense, row-major, in the layouts written beside each
 *     argument.  bf16 means IEEE bfloat16 bit patterns.  q, pools, cache,
 *     weights, out and workspace must be 16-byte aligned; block_table,
 *     context_lens and lse 4-byte aligned.  Misalignment returns
 *     PA_ERR_MISALIGNED before anything is launched.
 *   - Calls are asynchronous on `stream` (no host synchronisation) except
 *     pa_read_device_status.
 *   - Scores are scale * q.k in fp32; probabilities and accumulators are
 *     fp32; out is rounded to bf16 (round to nearest even); lse is the
 *     natural-log log-sum-exp of the scores in fp32, -inf for an empty row
 *     (whose out is 0).
 *   - Row b attends to logical tokens [lo, L) with L = context_lens[b] and
 *     lo = max(0, L - window) when window > 0 (the `window` most recent keys,
 *     current token included), else lo = 0.  Logical token t lives in
 *     physical page block_table[b][t / page_size], slot t % page_size.
 *     Table entries past a row's last visible page are never read.
 *   - Preconditions the host cannot check (they live in device memory):
 *     0 <= context_lens[b] <= max_context_len and every visited table entry
 *     in [0, num_pages).  A violation never traps: the kernel records a bit
 *     in the workspace's device status word (pa_read_device_status), clamps
 *     the length / skips the page, and the output of that row is unspecified.
 *   - num_splits, GQA: the visible keys of every (row, KV head) sequence,
 *     flattened row by row, are cut into that many equal contiguous shares,
 *     each handled by one CTA and merged in ascending order where a sequence
 *     spans several shares; 0 = automatic (one share per SM, at most 256),
 *     n in [1, 4096] = n shares; MLA the same, its sequences being (row, tile
 *     of 128 heads, half of the 512 latent columns) over the one latent cache
 *     row.  For a
 *     fixed num_splits (and fixed inputs) results are bitwise reproducible
 *     from run to run and independent of the physical page order; different
 *     split counts agree within rounding.
 *   - Workspace: at least pa_workspace_size(...) bytes of device memory for
 *     the same (kind, shape, max_context_len, page_size, num_splits).  Its
 *     contents need no initialisation and are overwritten by each call;
 *     calls sharing one workspace must be ordered on one stream.  The GQA
 *     workspace holds two fp32 partial results of 32 rows -- two 16-row tiles
 *     of query rows -- per share (32 KB per share at head_dim 128, about 8.5 MB
 *     in automatic mode) and two int32 tables with an entry per (row, KV head,
 *     tile) for up to 64 query positions (2 KB per (row, KV head)); it does
 *     not depend on the context lengths.  The MLA workspace holds two fp32 partial
 *     results of min(num_heads, 128) heads x 256 columns per share (256 KB
 *     per share for 128 heads, 64 MB in automatic mode), plus q_abs, q_lo and
 *     o_lat in bf16 (3.1 KB per (row, head)) and two int32 tables of where
 *     each (row, head tile, column half) sequence's pieces are (16 bytes per
 *     (row, tile of 128 heads)).
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARGUMENT = -1, /* a size <= 0 where one is needed, Hq % Hkv != 0, NULL pointer, ... */
  PA_ERR_UNSUPPORTED = -2,      /* head_dim not 64/128/256, page_size not an accepted power of two, ... */
  PA_ERR_MISALIGNED = -3,       /* a pointer breaks the alignment rule above */
  PA_ERR_WORKSPACE_TOO_SMALL = -4,
  PA_ERR_CUDA = -5              /* a CUDA runtime call or launch failed (cudaGetLastError is left set) */
} pa_status;

typedef enum { PA_KIND_GQA = 0, PA_KIND_MLA_ABSORBED = 1 } pa_kind;

/* Bits of the device status word (see pa_read_device_status). */
#define PA_DEV_BAD_PAGE 0x1u /* a visited block-table entry was outside [0, num_pages) */
#define PA_DEV_BAD_LEN 0x2u  /* a context length was < 0 or > max_context_len */
#define PA_DEV_TIMEOUT 0x4u  /* a bounded wait inside a kernel gave up (never expected at the default limit) */
#define PA_DEV_BAD_SLOT 0x8u /* a cache write named a slot at or past num_pages * page_size */

/*
 * Bytes of device workspace a call with these arguments needs.  For
 * PA_KIND_MLA_ABSORBED, num_q_heads is the head count and num_kv_heads /
 * head_dim are ignored.  Returns 0 for arguments the matching decode call
 * would reject.
 */
size_t pa_workspace_size(int kind, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_context_len, int page_size, int num_splits);

/*
 * GQA paged decode.
 *   q            [batch, num_q_heads, head_dim] bf16
 *   k_pool       [num_pages, page_size, num_kv_heads, head_dim] bf16
 *   v_pool       same shape as k_pool
 *   block_table  [batch, max_pages_per_seq] int32, logical page -> physical page
 *   context_lens [batch] int32
 *   out          [batch, num_q_heads, head_dim] bf16 (written)
 *   lse          [batch, num_q_heads] fp32 natural-log LSE (written), or NULL
 * Query head h reads KV head h / (num_q_heads / num_kv_heads).
 * head_dim in {64, 128, 256}; page_size a power of two in [8, 256];
 * max_pages_per_seq >= ceil(max_context_len / page_size); window <= 0 means
 * no window; num_splits in [0, 4096].  batch == 0 is a no-op returning PA_OK.
 */
int pa_decode_gqa(const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_table, const int32_t *context_lens, void *out, float *lse,
                  int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                  int num_pages, int max_pages_per_seq, int max_context_len, float scale,
                  int window, int num_splits, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/*
 * GQA multi-query (speculative-verify) decode: the Q newest tokens of every row
 * are queries, causal among themselves, and all of them share one walk over the
 * row's pages (vllm.cpp kernel-matrix, row KERNEL-ATTN-DFLASH-PAGED-BLOCK: the
 * block's queries causal within it over the paged cache; pegainfer PR #938's
 * verify launches).
 *   q            [batch, num_query, num_q_heads, head_dim] bf16
 *   out          [batch, num_query, num_q_heads, head_dim] bf16 (written)
 *   lse          [batch, num_query, num_q_heads] fp32 (written), or NULL
 *   context_lens [batch]: L, the row's length including its num_query new tokens
 * Query position i of a row sits at logical position L - num_query + i and
 * attends to keys [lo, L - num_query + 1 + i), lo = max(0, that - window) under a
 * window: the result of each (row, position) equals pa_decode_gqa on a row of
 * length L - num_query + 1 + i (0 or less: out = 0, lse = -inf).  Every other
 * argument, the workspace (same size as for pa_decode_gqa) and the error codes
 * are those of pa_decode_gqa; num_query in [1, 64] (1 is pa_decode_gqa).
 */
int pa_verify_gqa(const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_table, const int32_t *context_lens, void *out, float *lse,
                  int batch, int num_query, int num_q_heads, int num_kv_heads, int head_dim,
                  int page_size, int num_pages, int max_pages_per_seq, int max_context_len,
                  float scale, int window, int num_splits, void *workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/*
 * GQA decode and multi-query verify over an FP8 KV cache (vllm.cpp
 * kernel-matrix, row KERNEL-KV-QUANT, "FP8": the quantized form of the paged
 * cache).  The pools hold FP8 E4M3 codes, one byte per value (1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 NaN,
 * largest finite 448), and one float scale per pool turns a code into its
 * value: key = E4M3(code) * k_scale, value = E4M3(code) * v_scale.
 *   k_pool, v_pool [num_pages, page_size, num_kv_heads, head_dim] uint8 codes
 *   k_scale, v_scale finite and > 0 (else PA_ERR_INVALID_ARGUMENT)
 *   num_query    query positions per row as for pa_verify_gqa (1: decode, q of
 *                shape [batch, num_q_heads, head_dim])
 * Every other argument, the workspace (pa_workspace_size(PA_KIND_GQA, ...)),
 * the window and the error codes are those of pa_verify_gqa; head_dim in
 * {128, 256} (64: PA_ERR_UNSUPPORTED).  The codes enter FP8 tensor-core MMAs
 * unchanged.  Each query column (one head at one position) is scaled by a
 * power of two and split into two E4M3 terms, exact for every element above
 * 2^-10 of the column's largest magnitude.  The softmax weights are split into
 * two terms within 2^-8 relative.  Scores, softmax and accumulation are fp32.
 */
int pa_decode_gqa_fp8(const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *context_lens, void *out,
                      float *lse, int batch, int num_query, int num_q_heads, int num_kv_heads,
                      int head_dim, int page_size, int num_pages, int max_pages_per_seq,
                      int max_context_len, float scale, float k_scale, float v_scale, int window,
                      int num_splits, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * GQA decode and multi-query verify over an NVFP4 KV cache (vllm.cpp
 * kernel-matrix, row KERNEL-KV-QUANT, "Quantized KV cache, including FP8 and
 * NVFP4").  The pages name the format only; it is read as the published NVFP4
 * layout: 4-bit E2M1 values (1 sign, 2 exponent, 1 mantissa bit: magnitudes 0,
 * 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per block of 16 consecutive values
 * of a row, and one float scale per pool:
 *   key = E2M1(code) * E4M3(block scale) * k_scale   (values: v_scale)
 *   k_pool, v_pool [num_pages, page_size, num_kv_heads, R] uint8 rows,
 *                R = round_up(head_dim / 2 + head_dim / 16, 16) (48, 80, 144 at
 *                head_dim 64, 128, 256): head_dim / 2 bytes of code pairs (dim
 *                2i in the low nibble of byte i, 2i + 1 in the high nibble),
 *                then head_dim / 16 block-scale codes, then padding (not read)
 *   k_scale, v_scale finite and > 0 (else PA_ERR_INVALID_ARGUMENT)
 *   num_query    query positions per row as for pa_verify_gqa
 * Every other argument, the workspace (pa_workspace_size(PA_KIND_GQA, ...)),
 * the window and the error codes are those of pa_verify_gqa; head_dim in
 * {64, 128, 256}.  Each E2M1 value times its E4M3 block scale is an exact
 * bf16 value, so the keys and values enter bf16 tensor-core MMAs unrounded;
 * the pool scales multiply the fp32 scores and outputs.  A block scale that
 * decodes to NaN makes the values of its block NaN (as the format defines);
 * such a row is read only where it is attended.
 */
int pa_decode_gqa_nvfp4(const void *q, const void *k_pool, const void *v_pool,
                        const int32_t *block_table, const int32_t *context_lens, void *out,
                        float *lse, int batch, int num_query, int num_q_heads, int num_kv_heads,
                        int head_dim, int page_size, int num_pages, int max_pages_per_seq,
                        int max_context_len, float scale, float k_scale, float v_scale, int window,
                        int num_splits, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * MLA absorbed decode (DeepSeek-V2-style geometry: 128 nope + 64 rope query
 * dims, 512 latent + 64 rope cache dims, 128 value dims per head).
 *   q            [batch, num_heads, 192] bf16: q_nope (128) || q_rope (64)
 *   cache        [num_pages, page_size, 576] bf16: latent c (512) || rope key (64)
 *   w_uk         [num_heads, 128, 512] bf16, W_UK[h][d][j]: q_lat[j] = sum_d q_nope[d] W_UK[h][d][j]
 *   w_uv         [num_heads, 128, 512] bf16, W_UV[h][v][j]: o[v] = sum_j W_UV[h][v][j] o_lat[j]
 *   block_table, context_lens as for GQA (one latent head shared by all heads)
 *   out          [batch, num_heads, 128] bf16 (written)
 *   lse          [batch, num_heads] fp32 (written), or NULL
 * page_size a power of two in [8, 256]; num_splits as for GQA (shares, in [0, 4096]).
 */
int pa_decode_mla_absorbed(const void *q, const void *cache, const void *w_uk, const void *w_uv,
                           const int32_t *block_table, const int32_t *context_lens, void *out,
                           float *lse, int batch, int num_heads, int page_size, int num_pages,
                           int max_pages_per_seq, int max_context_len, float scale,
                           int num_splits, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * GQA paged decode without a caller-provided workspace.  The pages describe
 * no counterpart of this entry point: it exists for callers that cannot
 * allocate device memory when they call the decode (an engine whose device
 * memory is all held by its own pool, a plug-in that is handed only its input
 * and output pointers, a latency-critical path that must not pay for
 * cudaMalloc's possible device synchronisation).
 *
 * Arguments, layouts, results and error codes are those of pa_decode_gqa;
 * the workspace is a fixed device array of PA_NOALLOC_SCRATCH_BYTES inside
 * this library, which every GPU that loads the library keeps allocated until
 * the process exits.  Nothing is allocated or freed by the call.
 *   - A call whose pa_workspace_size(PA_KIND_GQA, ...) exceeds
 *     PA_NOALLOC_SCRATCH_BYTES returns PA_ERR_WORKSPACE_TOO_SMALL before any
 *     device work.  Automatic mode (num_splits 0) always fits; an explicit
 *     num_splits fits up to about 1000 shares at head_dim 128 (500 at 256).
 *   - The first call in a CUDA context (normally the device's primary
 *     context) looks up the array's device address in that context and
 *     caches it under the context's unique ID; make that first call before
 *     starting any stream capture on the device.  A context created later
 *     (after cudaDeviceReset, or one the caller makes current) has a new ID,
 *     so its first call looks the address up again.
 *   - All calls on a device share the one array.  Nothing in it has to start
 *     at zero (each call's split kernel writes every descriptor and partial
 *     slot the combine kernel then reads), but two calls that may overlap on
 *     the GPU race on it:
 *     order them on one stream, or use pa_decode_gqa with separate workspaces.
 *   - The array keeps the last call's contents; pa_read_device_status cannot
 *     reach it, so this entry point offers no device status word.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB per device */
int pa_decode_gqa_noalloc(const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_table, const int32_t *context_lens, void *out,
                          float *lse, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                          int page_size, int num_pages, int max_pages_per_seq, int max_context_len,
                          float scale, int window, int num_splits, cudaStream_t stream);

/*
 * Paged KV write: puts the keys and values of new tokens into their slots of
 * the paged pools, the step that precedes the decode (vllm.cpp kernel-matrix,
 * row KERNEL-KV-CACHE, ReshapeAndCache).
 *   k, v          [num_tokens, num_kv_heads, head_dim] bf16 (read)
 *   slot_mapping  [num_tokens] int64: token t goes to physical page
 *                 slot / page_size, slot slot % page_size; a negative slot is a
 *                 padding token and is skipped
 *   k_pool, v_pool [num_pages, page_size, num_kv_heads, head_dim] bf16 (written
 *                 at the named slots only; everything else is left untouched)
 *   status        optional device word (NULL: none); a slot at or past
 *                 num_pages * page_size is skipped and sets PA_DEV_BAD_SLOT
 * head_dim a multiple of 8 up to 1024.  The slots of one call must be distinct
 * (two tokens naming one slot leave either token's row there).  A pure copy:
 * the written bits equal the input bits.  num_tokens == 0 is a no-op.
 */
int pa_kv_write(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool, void *v_pool,
                int num_tokens, int num_kv_heads, int head_dim, int page_size, int num_pages,
                uint32_t *status, cudaStream_t stream);

/*
 * FP8 paged KV write: as pa_kv_write into FP8 E4M3 pools (the layout of
 * pa_decode_gqa_fp8): every bf16 value x of k (v) is stored as the E4M3 code
 * nearest to the fp32 quotient x / k_scale (x / v_scale), rounded to nearest
 * with ties to even, magnitudes above 448 saturating to 448 (NaN stays NaN).
 *   k_pool, v_pool [num_pages, page_size, num_kv_heads, head_dim] uint8 codes
 *   k_scale, v_scale finite and > 0 (else PA_ERR_INVALID_ARGUMENT)
 * head_dim a multiple of 16 up to 1024; k_pool and v_pool 16-byte aligned, k
 * and v 16-byte aligned.  slot_mapping, status and num_tokens as for
 * pa_kv_write.
 */
int pa_kv_write_fp8(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                    void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int page_size,
                    int num_pages, float k_scale, float v_scale, uint32_t *status,
                    cudaStream_t stream);

/*
 * NVFP4 paged KV write: as pa_kv_write into NVFP4 pools (the row layout of
 * pa_decode_gqa_nvfp4).  Each block of 16 consecutive bf16 values x of a
 * (token, head) row of k (v) is quantized in fp32 arithmetic, every step
 * correctly rounded, with s = k_scale (v_scale):
 *   block scale code c = E4M3((amax / s) / 6), amax = the largest |x| of the
 *                block; round to nearest, ties to even, saturating at 448; a
 *                NaN in the block gives the NaN code 0x7F
 *   value code   E2M1((x / s) / E4M3(c)), round to nearest, ties to even
 *                (the code with the even mantissa bit), magnitudes above 6
 *                saturating to 6, the sign bit taken from the quotient; every
 *                code of the block 0 where E4M3(c) is 0 or NaN
 *   k_pool, v_pool [num_pages, page_size, num_kv_heads, R] uint8 rows; the whole
 *                row of a named slot is written, its padding bytes as zeros
 *   k_scale, v_scale finite and > 0 (else PA_ERR_INVALID_ARGUMENT)
 * head_dim in {64, 128, 256} (else PA_ERR_UNSUPPORTED); k and v 16-byte
 * aligned, the pools 16-byte aligned.  slot_mapping, status and num_tokens as
 * for pa_kv_write.
 */
int pa_kv_write_nvfp4(const void *k, const void *v, const int64_t *slot_mapping, void *k_pool,
                      void *v_pool, int num_tokens, int num_kv_heads, int head_dim, int page_size,
                      int num_pages, float k_scale, float v_scale, uint32_t *status,
                      cudaStream_t stream);

/*
 * MLA cache write: the 576-wide cache row of each new token is its latent
 * (512) followed by its rope key (64) (vllm.cpp kernel-matrix, row
 * KERNEL-KV-CACHE, ConcatAndCacheMla).
 *   c_lat   [num_tokens, 512] bf16, k_rope [num_tokens, 64] bf16 (read)
 *   cache   [num_pages, page_size, 576] bf16 (written at the named slots only)
 * slot_mapping and status as for pa_kv_write.
 */
int pa_mla_cache_write(const void *c_lat, const void *k_rope, const int64_t *slot_mapping, void *cache,
                       int num_tokens, int page_size, int num_pages, uint32_t *status,
                       cudaStream_t stream);

/* Static text for a pa_status value (never NULL). */
const char *pa_status_string(int status);

/*
 * Synchronises `stream`, then copies the device status word of `workspace`
 * (as left by the last call that used it) into *out_bits (PA_DEV_* bits).
 * Returns PA_ERR_CUDA if the copy or the synchronisation fails.
 */
int pa_read_device_status(const void *workspace, cudaStream_t stream, uint32_t *out_bits);

/*
 * Measurement hook: on the calling host thread, subsequent decode calls
 * record `before_main` just before and `after_main` just after the launch of
 * their dominant kernel (the split-KV attention kernel), on the call's
 * stream.  Pass NULL, NULL to switch it off.  Events are owned by the caller.
 */
int pa_set_profile_events(cudaEvent_t before_main, cudaEvent_t after_main);

/* Number of kernel launches the last decode call on this host thread issued. */
int pa_last_launch_count(void);

/*
 * Limit of the waits on the stage ring of the GQA split-KV kernels
 * (pa_decode_gqa, pa_verify_gqa, pa_decode_gqa_fp8, pa_decode_gqa_nvfp4 and the
 * no-alloc decode),
 * in nanoseconds of the device's global timer, for later calls from the
 * calling host thread.  The pages have no counterpart: it is a diagnostic
 * for checking that the kernels leave cleanly when a wait does not complete.
 * The default, PA_DEFAULT_WAIT_LIMIT_NS (1 s), is far beyond any legal wait;
 * 0 makes a warp give up at the first wait it finds incomplete.
 *
 * A warp whose wait passes the limit records PA_DEV_TIMEOUT in the call's
 * status word and gives up its work while keeping the ring's protocol: the
 * producer issues no further copy and ends the ring once the slot it waited
 * for is free; a consumer computes nothing more but still releases every
 * stage and meets every barrier.  Copies already in flight land first
 * (waiting up to another second), so no CTA ends with a copy in flight or
 * leaves a warp waiting.  The call still returns normally, but its out and
 * lse are unspecified.  The next call with a sufficient limit is
 * unaffected.  The MLA kernels always use the default.  A call at the
 * default limit runs kernels compiled with the 1 s bound fixed; a call with
 * any other limit runs the same kernels compiled with it as an argument.
 * Always returns PA_OK.
 */
#define PA_DEFAULT_WAIT_LIMIT_NS 1000000000ull
int pa_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * The CUDA runtime error (a cudaError_t value) behind the most recent
 * PA_ERR_CUDA returned by any entry point on the calling thread, and its
 * text; cudaSuccess (0) and "no error" if no call on this thread has returned
 * PA_ERR_CUDA.  Calls that succeed leave it unchanged.  The pages describe no
 * counterpart: it is diagnostics for the boundary's PA_ERR_CUDA code.
 */
int pa_last_cuda_error(void);
const char *pa_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
