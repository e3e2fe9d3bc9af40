/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library; it reads the same seeded input bits and nothing else.
 *
 * What it computes (the pages give no formula; they name the pieces):
 *   - the paged KV cache: K and V pools shaped [pages, page_size, Hkv, D],
 *     a per-row context length and a block table mapping logical page ->
 *     physical page (vllm.cpp kernel-matrix, rows KERNEL-ATTN-PAGED and
 *     KERNEL-ATTN-DFLASH-PAGED-BLOCK);
 *   - GQA grouping: query heads share one KV head (vllm.cpp PR #425
 *     "head_dim-128 arm for the warp-split-KV decode kernel", the GQA
 *     carve-out paragraph; vllm.cpp PR #49 "flip decode GQA group-swap
 *     default ON", mechanism paragraph).  Reading: contiguous grouping,
 *     kv head = h / (Hq / Hkv);
 *   - the optional sliding window (PR #425 limitations list, the HasWindow
 *     arm; kernel-matrix row KERNEL-ATTN-DFLASH-BLOCK, "causal-within-window").
 *     Reading: a row of length L attends to keys t in [max(0, L - W), L);
 *   - softmax(q . K^T * scale) . V per query head, and its log-sum-exp.
 *     The oracle deliberately uses the plain two-pass form (max, then sum),
 *     not the online recurrence the kernels use;
 *   - the LSE merge of split partials (kernel-matrix row
 *     KERNEL-ATTN-MLA-SPARSE: fixed ascending split merge, empty splits
 *     carry -inf);
 *   - MLA absorbed decode, the seven-step schedule of pegainfer PR #938
 *     "warp-cooperative two-pass MLA absorbed decode kernel" (Schedule
 *     section, steps 1-7) WITHOUT its bf16 landings: q_lat = q_nope . W_UK,
 *     scores over the 576-wide latent||rope cache, softmax, o_lat = sum p c,
 *     o = W_UV . o_lat.
 *
 * Inputs are raw bf16 bit patterns widened exactly to double.  Every sum is
 * a plain left-to-right loop in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int pa_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Physical page holding logical token t of row b, or -1 if the table entry is
 * outside the pool. */
static int64_t page_of(const int32_t *block_table, int max_pages_per_seq, int num_pages,
                       int page_size, int b, int64_t t) {
  int64_t lp = t / page_size;
  if (lp >= max_pages_per_seq) return -1;
  int32_t p = block_table[(int64_t)b * max_pages_per_seq + lp];
  if (p < 0 || p >= num_pages) return -1;
  return p;
}

/* Attention of query head h of row b over logical tokens [t0, t1).
 * Two passes: scores into s[], then max / sum / weighted V. */
static int gqa_one(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                   const int32_t *block_table, int Hq, int Hkv, int D, int P, int num_pages,
                   int max_pages_per_seq, double scale, int b, int h, int64_t t0, int64_t t1,
                   double *s, double *o, double *lse) {
  int G = Hq / Hkv;
  int g = h / G; /* contiguous grouping */
  const uint16_t *qh = q + ((int64_t)b * Hq + h) * D;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (t1 <= t0) {
    *lse = -INFINITY;
    return ORACLE_OK;
  }
  /* pass 1: raw scores */
  for (int64_t t = t0; t < t1; ++t) {
    int64_t p = page_of(block_table, max_pages_per_seq, num_pages, P, b, t);
    if (p < 0) return ORACLE_EINVAL;
    int64_t slot = t % P;
    const uint16_t *kr = k_pool + ((p * P + slot) * Hkv + g) * D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += bf16_to_double(qh[d]) * bf16_to_double(kr[d]);
    s[t - t0] = scale * dot;
  }
  double m = -INFINITY;
  for (int64_t t = t0; t < t1; ++t)
    if (s[t - t0] > m) m = s[t - t0];
  double Z = 0.0;
  for (int64_t t = t0; t < t1; ++t) Z += exp(s[t - t0] - m);
  /* pass 2: probabilities times V */
  for (int64_t t = t0; t < t1; ++t) {
    int64_t p = page_of(block_table, max_pages_per_seq, num_pages, P, b, t);
    int64_t slot = t % P;
    const uint16_t *vr = v_pool + ((p * P + slot) * Hkv + g) * D;
    double pt = exp(s[t - t0] - m) / Z;
    for (int d = 0; d < D; ++d) o[d] += pt * bf16_to_double(vr[d]);
  }
  *lse = m + log(Z);
  return ORACLE_OK;
}

static int gqa_check(int B, int Hq, int Hkv, int D, int P, int num_pages, int max_pages_per_seq) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || num_pages <= 0 ||
      max_pages_per_seq <= 0)
    return ORACLE_EINVAL;
  if (Hq % Hkv != 0) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Core over explicit (row, head, token span) items; shared by the two entry
 * points below. */
static int gqa_items(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                     const int32_t *block_table, int B, int Hq, int Hkv, int D, int P,
                     int num_pages, int max_pages_per_seq, double scale, int n_items,
                     const int32_t *items_b, const int32_t *items_h, const int64_t *items_t0,
                     const int64_t *items_t1, double *out_o, double *out_lse, int nthreads) {
  int rc = gqa_check(B, Hq, Hkv, D, P, num_pages, max_pages_per_seq);
  if (rc) return rc;
  int64_t span_max = 1;
  for (int i = 0; i < n_items; ++i) {
    if (items_b[i] < 0 || items_b[i] >= B || items_h[i] < 0 || items_h[i] >= Hq)
      return ORACLE_EINVAL;
    if (items_t0[i] < 0) return ORACLE_EINVAL;
    if (items_t1[i] - items_t0[i] > span_max) span_max = items_t1[i] - items_t0[i];
  }
  int err = ORACLE_OK;
  if (nthreads <= 0) nthreads = pa_oracle_num_threads();
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)span_max);
    if (!s) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < n_items; ++i) {
        int r = gqa_one(q, k_pool, v_pool, block_table, Hq, Hkv, D, P, num_pages,
                        max_pages_per_seq, scale, items_b[i], items_h[i], items_t0[i],
                        items_t1[i], s, out_o + (int64_t)i * D, out_lse + i);
        if (r) {
#pragma omp atomic write
          err = r;
        }
      }
      free(s);
    }
  }
  return err;
}

/*
 * GQA decode oracle.  For each item i, query head items_h[i] of row
 * items_b[i] attends to the visible keys of its row: all L keys, or the W most
 * recent ones when window W > 0.  out_o is [n_items, D], out_lse [n_items]
 * (natural log; -inf for an empty row).
 */
int pa_oracle_gqa(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                  const int32_t *block_table, const int32_t *context_lens, int B, int Hq,
                  int Hkv, int D, int P, int num_pages, int max_pages_per_seq, double scale,
                  int window, int n_items, const int32_t *items_b, const int32_t *items_h,
                  double *out_o, double *out_lse, int nthreads) {
  if (n_items < 0 || B <= 0) return ORACLE_EINVAL;
  int64_t *t0 = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_items + 1));
  int64_t *t1 = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_items + 1));
  if (!t0 || !t1) {
    free(t0);
    free(t1);
    return ORACLE_ENOMEM;
  }
  int rc = ORACLE_OK;
  for (int i = 0; i < n_items; ++i) {
    if (items_b[i] < 0 || items_b[i] >= B) {
      rc = ORACLE_EINVAL;
      break;
    }
    int64_t L = context_lens[items_b[i]];
    if (L < 0) {
      rc = ORACLE_EINVAL;
      break;
    }
    t1[i] = L;
    t0[i] = (window > 0 && L > window) ? L - window : 0;
  }
  if (rc == ORACLE_OK)
    rc = gqa_items(q, k_pool, v_pool, block_table, B, Hq, Hkv, D, P, num_pages,
                   max_pages_per_seq, scale, n_items, items_b, items_h, t0, t1, out_o, out_lse,
                   nthreads);
  free(t0);
  free(t1);
  return rc;
}

/* Same attention over an explicit logical token span [t0, t1) per item (the
 * partial a split of the KV sequence computes). */
int pa_oracle_gqa_span(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                       const int32_t *block_table, int B, int Hq, int Hkv, int D, int P,
                       int num_pages, int max_pages_per_seq, double scale, int n_items,
                       const int32_t *items_b, const int32_t *items_h, const int64_t *items_t0,
                       const int64_t *items_t1, double *out_o, double *out_lse, int nthreads) {
  return gqa_items(q, k_pool, v_pool, block_table, B, Hq, Hkv, D, P, num_pages,
                   max_pages_per_seq, scale, n_items, items_b, items_h, items_t0, items_t1,
                   out_o, out_lse, nthreads);
}

/*
 * Merge of split partials (o_s normalised within its split, lse_s its
 * log-sum-exp) in ascending split order:
 *   lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
 * Splits with lse_s = -inf are empty and contribute nothing; if every split
 * is empty the result is o = 0, lse = -inf.
 */
int pa_oracle_merge(int n_parts, int D, const double *parts_o, const double *parts_lse,
                    double *out_o, double *out_lse) {
  if (n_parts < 0 || D <= 0) return ORACLE_EINVAL;
  double m = -INFINITY;
  for (int s = 0; s < n_parts; ++s)
    if (parts_lse[s] > m) m = parts_lse[s];
  for (int d = 0; d < D; ++d) out_o[d] = 0.0;
  if (m == -INFINITY) {
    *out_lse = -INFINITY;
    return ORACLE_OK;
  }
  double Z = 0.0;
  for (int s = 0; s < n_parts; ++s)
    if (parts_lse[s] != -INFINITY) Z += exp(parts_lse[s] - m);
  double lse = m + log(Z);
  for (int s = 0; s < n_parts; ++s) {
    if (parts_lse[s] == -INFINITY) continue;
    double w = exp(parts_lse[s] - lse);
    for (int d = 0; d < D; ++d) out_o[d] += w * parts_o[(int64_t)s * D + d];
  }
  *out_lse = lse;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* MLA absorbed decode.                                                      */
/* ------------------------------------------------------------------------ */
#define MLA_NOPE 128
#define MLA_ROPE 64
#define MLA_QDIM (MLA_NOPE + MLA_ROPE)
#define MLA_LAT 512
#define MLA_CDIM (MLA_LAT + MLA_ROPE)
#define MLA_VDIM 128

/*
 * For each item (row b, head h), with L = context_lens[b]:
 *   1. q_lat[j] = sum_d q_nope[d] * W_UK[h][d][j]          (j < 512)
 *   2. s_t = scale * (sum_j q_lat[j] c_t[j] + sum_r q_rope[r] c_t[512 + r])
 *   3. m = max_t s_t, Z = sum_t exp(s_t - m), p_t = exp(s_t - m) / Z
 *   4. o_lat[j] = sum_t p_t c_t[j]                          (j < 512)
 *   5. o[dv] = sum_j W_UV[h][dv][j] o_lat[j]                (dv < 128)
 *   lse = m + log Z.
 * q is [B, H, 192] (nope || rope), cache [pages, P, 576] (latent || rope key),
 * W_UK and W_UV are [H, 128, 512].  out_o [n, 128], out_lse [n]; out_qlat and
 * out_olat ([n, 512]) are optional intermediates (may be NULL).
 */
int pa_oracle_mla(const uint16_t *q, const uint16_t *cache, const uint16_t *w_uk,
                  const uint16_t *w_uv, const int32_t *block_table, const int32_t *context_lens,
                  int B, int H, int P, int num_pages, int max_pages_per_seq, double scale,
                  int n_items, const int32_t *items_b, const int32_t *items_h, double *out_o,
                  double *out_lse, double *out_qlat, double *out_olat, int nthreads) {
  if (B <= 0 || H <= 0 || P <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 || n_items < 0)
    return ORACLE_EINVAL;
  int64_t Lmax = 1;
  for (int i = 0; i < n_items; ++i) {
    if (items_b[i] < 0 || items_b[i] >= B || items_h[i] < 0 || items_h[i] >= H)
      return ORACLE_EINVAL;
    if (context_lens[items_b[i]] < 0) return ORACLE_EINVAL;
    if (context_lens[items_b[i]] > Lmax) Lmax = context_lens[items_b[i]];
  }
  int err = ORACLE_OK;
  if (nthreads <= 0) nthreads = pa_oracle_num_threads();
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
    double qlat[MLA_LAT], olat[MLA_LAT];
    if (!s) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int i = 0; i < n_items; ++i) {
        int b = items_b[i], h = items_h[i];
        int64_t L = context_lens[b];
        const uint16_t *qn = q + ((int64_t)b * H + h) * MLA_QDIM;
        const uint16_t *qr = qn + MLA_NOPE;
        const uint16_t *wk = w_uk + (int64_t)h * MLA_NOPE * MLA_LAT;
        const uint16_t *wv = w_uv + (int64_t)h * MLA_VDIM * MLA_LAT;
        /* step 1 */
        for (int j = 0; j < MLA_LAT; ++j) {
          double acc = 0.0;
          for (int d = 0; d < MLA_NOPE; ++d)
            acc += bf16_to_double(qn[d]) * bf16_to_double(wk[(int64_t)d * MLA_LAT + j]);
          qlat[j] = acc;
        }
        /* step 2 */
        int bad = 0;
        for (int64_t t = 0; t < L && !bad; ++t) {
          int64_t p = page_of(block_table, max_pages_per_seq, num_pages, P, b, t);
          if (p < 0) {
            bad = 1;
            break;
          }
          const uint16_t *c = cache + (p * P + t % P) * MLA_CDIM;
          double dot = 0.0;
          for (int j = 0; j < MLA_LAT; ++j) dot += qlat[j] * bf16_to_double(c[j]);
          for (int r = 0; r < MLA_ROPE; ++r)
            dot += bf16_to_double(qr[r]) * bf16_to_double(c[MLA_LAT + r]);
          s[t] = scale * dot;
        }
        if (bad) {
#pragma omp atomic write
          err = ORACLE_EINVAL;
          continue;
        }
        /* steps 3-4 */
        for (int j = 0; j < MLA_LAT; ++j) olat[j] = 0.0;
        double m = -INFINITY, Z = 0.0, lse = -INFINITY;
        if (L > 0) {
          for (int64_t t = 0; t < L; ++t)
            if (s[t] > m) m = s[t];
          for (int64_t t = 0; t < L; ++t) Z += exp(s[t] - m);
          for (int64_t t = 0; t < L; ++t) {
            int64_t p = page_of(block_table, max_pages_per_seq, num_pages, P, b, t);
            const uint16_t *c = cache + (p * P + t % P) * MLA_CDIM;
            double pt = exp(s[t] - m) / Z;
            for (int j = 0; j < MLA_LAT; ++j) olat[j] += pt * bf16_to_double(c[j]);
          }
          lse = m + log(Z);
        }
        /* step 5 */
        double *o = out_o + (int64_t)i * MLA_VDIM;
        for (int dv = 0; dv < MLA_VDIM; ++dv) {
          double acc = 0.0;
          for (int j = 0; j < MLA_LAT; ++j)
            acc += bf16_to_double(wv[(int64_t)dv * MLA_LAT + j]) * olat[j];
          o[dv] = acc;
        }
        out_lse[i] = lse;
        if (out_qlat) memcpy(out_qlat + (int64_t)i * MLA_LAT, qlat, sizeof qlat);
        if (out_olat) memcpy(out_olat + (int64_t)i * MLA_LAT, olat, sizeof olat);
      }
      free(s);
    }
  }
  return err;
}
