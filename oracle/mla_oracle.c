/*
 * mla_oracle.c -- plain float64 CPU oracle for absorbed-form MLA decode and
 * causal multi-token speculative verification over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA library: it is written from the definitions on the
 * pages, slowly and directly, so that a reader can check it by eye.
 *
 * Page abbreviations used in the citations below:
 *   [vLLM #51705]  "ROCm AITER MLA supports causal multi-token speculative
 *                  verification under DCP" (vLLM pull request digest)
 *   [sglang #34432] "[AMD][DCP 1/N] add dcp support for aiter backend"
 *                  (sglang pull request digest)
 *   [vLLM #51011]  "fix silent wrong decoding of the fp8 KV cache on the ROCm
 *                  AITER MLA backend" (vLLM pull request digest)
 *
 * Arithmetic: every score, exponential, sum and output is a C double.  Cached
 * values are converted exactly (bf16 and e4m3 are subsets of double).  Lengths
 * and indices are int32/int64.  Compiled with -ffp-contract=off so that no
 * fused multiply-add changes the rounding between machines.
 *
 * Parity status: every function below is pinned by tests (closed forms,
 * invariants, brute force on tiny inputs, the e4m3 codes of a library
 * routine); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_DK 576 /* q / K width: 512 latent (k_nope) + 64 rope (k_pe) */
#define ORC_DV 512 /* V width: the 512-d latent k_nope                   */

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_QLEN 2
#define ORC_ERR_INDPTR 3
#define ORC_ERR_BLOCK 4
#define ORC_ERR_UNSUPPORTED 5
#define ORC_ERR_NOMEM 6
#define ORC_ERR_SLOT 7

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Sub-page size.  [vLLM #51705, 实现拆解 3 and the _segmented_mla_page_size
 * snippet]: the largest power of two that divides the physical block size,
 * capped at 128; block_size must be positive.  Returns -1 otherwise.        */
int oracle_page_size(int block_size) {
  if (block_size <= 0) return -1;
  int p = 1;
  /* grow p while 2p still divides block_size */
  while (block_size % (2 * p) == 0) p = 2 * p;
  if (p > 128) p = 128;
  return p;
}

/* ------------------------------------------------------------------------ */
/* Row plan.  [vLLM #51705, 实现拆解 2 and the _build_dcp_verify_row_view
 * snippet]: verify row t of a request with seq_len L and qlen rows sees the
 * global positions [0, L - qlen + t] inclusive (its own token included), i.e.
 * a window of L - qlen + 1 + t tokens.  The qlen new tokens are already in
 * the cache, so 1 <= qlen <= L is required.                                  */
int oracle_plan_rows(int num_reqs, const int32_t *seq_lens,
                     const int32_t *qo_indptr, int num_rows, int32_t *row_len,
                     int32_t *row_req, int32_t *row_t) {
  if (num_reqs < 0 || qo_indptr[0] != 0) return ORC_ERR_INDPTR;
  if (qo_indptr[num_reqs] > num_rows) return ORC_ERR_INDPTR;
  for (int b = 0; b < num_reqs; b++) {
    int qlen = qo_indptr[b + 1] - qo_indptr[b];
    int L = seq_lens[b];
    if (qlen < 1 || qlen > L) return ORC_ERR_QLEN;
    for (int t = 0; t < qlen; t++) {
      int i = qo_indptr[b] + t;
      int last_visible = L - qlen + t; /* inclusive end of the window */
      row_len[i] = last_visible + 1;
      row_req[i] = b;
      row_t[i] = t;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Round-robin (interleave 1) shard-local count.  [vLLM #51705, the
 * _build_dcp_verify_row_view snippet]: for a window of w global positions and
 * rank r of W, the number of positions the rank holds is floor((w-1-r)/W)+1
 * when that is non-negative, else 0.  [sglang #34432, key snippet]: local
 * index j of rank r is global position g(j) = j*W + r.                       */
int64_t oracle_rr_local_len(int64_t w, int world_size, int rank) {
  int64_t top = w - 1 - rank;
  if (top < 0) return 0;
  return top / world_size + 1; /* top >= 0, so C division is floor */
}

/* Round-robin with interleave I (the pages support only I = 1 and reject
 * the rest as unverified [vLLM #51705, 实现拆解 1]; the reading used here is
 * the plain generalisation of g(j) = j*W + r): the global positions are cut
 * into runs of I consecutive positions, dealt to the ranks in turn, so
 * position g belongs to rank (g div I) mod W, at local index
 * (g div (I*W)) * I + g mod I.  For a window of w positions, rank r holds
 * I per full cycle of I*W positions plus its part of the last, partial
 * cycle.  I = 1 reduces to oracle_rr_local_len.                              */
int64_t oracle_il_local_len(int64_t w, int world_size, int rank, int interleave) {
  if (w <= 0) return 0;
  const int64_t cycle = (int64_t)interleave * world_size;
  int64_t rem = w % cycle - (int64_t)rank * interleave;
  if (rem < 0) rem = 0;
  if (rem > interleave) rem = interleave;
  return (w / cycle) * interleave + rem;
}
int oracle_il_owner(int64_t g, int world_size, int interleave) {
  return (int)((g / interleave) % world_size);
}
int64_t oracle_il_local_index(int64_t g, int world_size, int interleave) {
  return (g / ((int64_t)interleave * world_size)) * interleave + g % interleave;
}

/* Shard row view: each verify row keeps its own shard-local length, counted
 * from the row's GLOBAL window (never "local length minus an offset").
 * [vLLM #51705, 实现拆解 2].  interleave 1 is the pages' form; other values
 * follow the generalisation above.                                          */
int oracle_shard_row_view(int num_rows, const int32_t *row_len_global,
                          int world_size, int rank, int interleave,
                          int32_t *row_len_local) {
  if (interleave < 1) return ORC_ERR_UNSUPPORTED;
  if (world_size < 1 || rank < 0 || rank >= world_size) return ORC_ERR_ARG;
  for (int i = 0; i < num_rows; i++)
    row_len_local[i] = interleave == 1
                           ? (int32_t)oracle_rr_local_len(row_len_global[i], world_size, rank)
                           : (int32_t)oracle_il_local_len(row_len_global[i], world_size, rank, interleave);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Sub-page table.  [vLLM #51705, 实现拆解 3, _fill_dcp_verify_page_table]:
 * the cache is reinterpreted as pages of P tokens; physical block `blk` of
 * block_size tokens holds the R = block_size / P sub-pages blk*R .. blk*R+R-1.
 * Local page p of a request therefore is block_table[p / R] * R + p % R.
 * Entries past the request's last page are -1.  kv_len[b] is the number of
 * tokens of request b in this table's address space.                         */
int oracle_subpage_table(int num_reqs, const int32_t *kv_len,
                         const int32_t *block_table, int bt_stride,
                         int num_blocks, int block_size, int32_t *sp_table,
                         int sp_stride) {
  int P = oracle_page_size(block_size);
  if (P < 0) return ORC_ERR_ARG;
  int R = block_size / P;
  for (int b = 0; b < num_reqs; b++) {
    int n_pages = (kv_len[b] + P - 1) / P;
    if (n_pages > sp_stride) return ORC_ERR_ARG;
    for (int p = 0; p < sp_stride; p++) {
      int32_t v = -1;
      if (p < n_pages) {
        int blk = block_table[(int64_t)b * bt_stride + p / R];
        if (blk < 0 || blk >= num_blocks) return ORC_ERR_BLOCK;
        v = blk * R + p % R;
      }
      sp_table[(int64_t)b * sp_stride + p] = v;
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* fp8 e4m3 (OCP "fn" variant: no infinities, S.1111.111 is NaN, max 448).
 * Value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * (m/8) for
 * e == 0.  The cache holds e4m3 codes and one per-tensor float scale
 * [sglang #34432, key snippet: kv_scale=_resolve_fp8_kv_scale_float(...)];
 * [vLLM #51011 describes the fp8 cache path].                               */
double oracle_e4m3_to_double(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* bf16 bit pattern -> double (exact: bf16 is the top half of a float). */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Cached element d of cache row `slot`, as a double, scale applied. */
static double cached_value(const void *kv, int kv_dtype, int64_t slot, int d,
                           double kv_scale) {
  if (kv_dtype == 0)
    return bf16_bits_to_double(((const uint16_t *)kv)[slot * ORC_DK + d]);
  return oracle_e4m3_to_double(((const uint8_t *)kv)[slot * ORC_DK + d]) *
         kv_scale;
}

static int request_of_row(int num_reqs, const int32_t *qo_indptr, int row) {
  for (int b = 0; b < num_reqs; b++)
    if (row >= qo_indptr[b] && row < qo_indptr[b + 1]) return b;
  return -1;
}

/* Physical cache row of token j of request b, walking the BLOCK table
 * directly (block j / block_size, offset j % block_size).  Independent of the
 * sub-page concept on purpose.                                               */
static int64_t slot_of_token(const int32_t *block_table, int bt_stride, int b,
                             int64_t j, int block_size) {
  int32_t blk = block_table[(int64_t)b * bt_stride + j / block_size];
  if (blk < 0) return -1;
  return (int64_t)blk * block_size + j % block_size;
}

/* ------------------------------------------------------------------------ */
/* Attention over an explicit per-row visible length, the plain definition.
 *
 * Absorbed-form MLA [sglang #34432, key snippet forward_mla_rocm.py]:
 *   q = cat(q_nope_out (512), q_pe (64)) per head,
 *   k = cat(k_nope (512 latent), k_pe (64 rope)) per cached token,
 *   v = k_nope, the first 512 entries of the cached row.
 * For row i (request b) and head h, with visible tokens j in [0, n_i):
 *   s_j  = sm_scale * sum_{d<576} q[i,h,d] * khat[j,d]
 *   out  = sum_j exp(s_j - m) vhat[j,:] / sum_j exp(s_j - m),  m = max s_j
 *   lse  = m + ln sum_j exp(s_j - m)      (natural log [sglang #34432,
 *          评论区精华 4: DCP LSE must be base e])
 * An empty row (n_i = 0) gives out = 0 and lse = -inf.
 *
 * Selection: if n_sel < 0 every (row, head) is computed and out/lse are laid
 * out [num_rows, H, 512] / [num_rows, H]; otherwise only the listed pairs, in
 * order, into out[n_sel, 512] / lse[n_sel].  Returns 0 or an error code.      */
int oracle_attention(int num_reqs, int num_heads, const int32_t *qo_indptr,
                     const int32_t *row_len, const uint16_t *q, const void *kv,
                     int kv_dtype, int64_t kv_rows, double kv_scale,
                     double sm_scale, const int32_t *block_table,
                     int bt_stride, int block_size, int n_sel,
                     const int32_t *sel_row, const int32_t *sel_head,
                     double *out, double *lse) {
  int num_rows = qo_indptr[num_reqs];
  int64_t n_items = n_sel < 0 ? (int64_t)num_rows * num_heads : n_sel;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < n_items; it++) {
    int row = n_sel < 0 ? (int)(it / num_heads) : sel_row[it];
    int h = n_sel < 0 ? (int)(it % num_heads) : sel_head[it];
    double *o = out + it * ORC_DV;
    int b = request_of_row(num_reqs, qo_indptr, row);
    int64_t n = row_len[row];
    if (b < 0 || n < 0) {
#pragma omp atomic write
      err = ORC_ERR_ARG;
      continue;
    }
    for (int d = 0; d < ORC_DV; d++) o[d] = 0.0;
    if (n == 0) {
      lse[it] = -INFINITY;
      continue;
    }
    const uint16_t *qv = q + ((int64_t)row * num_heads + h) * ORC_DK;
    double qd[ORC_DK];
    for (int d = 0; d < ORC_DK; d++) qd[d] = bf16_bits_to_double(qv[d]);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) {
#pragma omp atomic write
      err = ORC_ERR_NOMEM;
      continue;
    }
    /* scores */
    double m = -INFINITY;
    int bad = 0;
    for (int64_t j = 0; j < n; j++) {
      int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
      if (slot < 0 || slot >= kv_rows) {
        bad = 1;
        break;
      }
      double acc = 0.0;
      for (int d = 0; d < ORC_DK; d++)
        acc += qd[d] * cached_value(kv, kv_dtype, slot, d, kv_scale);
      s[j] = sm_scale * acc;
      if (s[j] > m) m = s[j];
    }
    if (bad) {
      free(s);
#pragma omp atomic write
      err = ORC_ERR_BLOCK;
      continue;
    }
    /* softmax-weighted sum of V */
    double denom = 0.0;
    for (int64_t j = 0; j < n; j++) {
      int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
      double e = exp(s[j] - m);
      denom += e;
      for (int d = 0; d < ORC_DV; d++)
        o[d] += e * cached_value(kv, kv_dtype, slot, d, kv_scale);
    }
    for (int d = 0; d < ORC_DV; d++) o[d] /= denom;
    lse[it] = m + log(denom);
    free(s);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Split-K segment partials in the pages' base-2 convention.
 * [vLLM #51705, 实现拆解 4 and the merge_mla_segments_triton snippet]:
 * the segmented kernel splits a sequence into NUM_SEGMENTS pieces of
 * tiles_per_segment = cdiv(seq_len, NUM_SEGMENTS * TILE_SIZE) tiles, with
 * TILE_SIZE the sub-page size P [实现拆解 3]; each segment keeps its local
 * max (base 2), its exp2 sum and its output.  Reading taken here: the
 * partition length is the longest row of the request (rows of one request
 * share the segment boundaries); a row's segment holds the tokens of the
 * segment's range that the row can see.  For each (row, head, segment):
 *   x_j   = s_j * log2(e)
 *   m_s   = max_j x_j over the segment's visible tokens (-inf if none)
 *   l_s   = sum_j 2^(x_j - m_s)                          (0 if none)
 *   acc_s = sum_j 2^(x_j - m_s) vhat[j,:]  (unnormalised; 0 if none)
 * Output layout: acc [num_rows, H, S, 512], m and l [num_rows, H, S]; only
 * n_sel < 0 (all pairs) is supported.                                        */
int oracle_segment_partials(int num_reqs, int num_heads,
                            const int32_t *qo_indptr, const int32_t *row_len,
                            const uint16_t *q, const void *kv, int kv_dtype,
                            int64_t kv_rows, double kv_scale, double sm_scale,
                            const int32_t *block_table, int bt_stride,
                            int block_size, int num_segments, int tile_size,
                            double *acc, double *mx, double *sm) {
  const double LOG2E = 1.0 / log(2.0);
  int num_rows = qo_indptr[num_reqs];
  int S = num_segments;
  int err = ORC_OK;
  if (S < 1 || tile_size < 1) return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < (int64_t)num_rows * num_heads; it++) {
    int row = (int)(it / num_heads);
    int h = (int)(it % num_heads);
    int b = request_of_row(num_reqs, qo_indptr, row);
    if (b < 0) {
#pragma omp atomic write
      err = ORC_ERR_ARG;
      continue;
    }
    /* partition length: the longest row of the request */
    int64_t group_len = 0;
    for (int r = qo_indptr[b]; r < qo_indptr[b + 1]; r++)
      if (row_len[r] > group_len) group_len = row_len[r];
    int64_t tps = (group_len + (int64_t)S * tile_size - 1) /
                  ((int64_t)S * tile_size);
    const uint16_t *qv = q + ((int64_t)row * num_heads + h) * ORC_DK;
    double qd[ORC_DK];
    for (int d = 0; d < ORC_DK; d++) qd[d] = bf16_bits_to_double(qv[d]);
    for (int s = 0; s < S; s++) {
      int64_t base = it * S + s;
      double *a = acc + base * ORC_DV;
      for (int d = 0; d < ORC_DV; d++) a[d] = 0.0;
      mx[base] = -INFINITY;
      sm[base] = 0.0;
      int64_t lo = (int64_t)s * tps * tile_size;
      int64_t hi = lo + tps * tile_size;
      if (hi > row_len[row]) hi = row_len[row];
      if (lo >= hi) continue;
      double *x = (double *)malloc(sizeof(double) * (size_t)(hi - lo));
      if (!x) {
#pragma omp atomic write
        err = ORC_ERR_NOMEM;
        break;
      }
      double m = -INFINITY;
      for (int64_t j = lo; j < hi; j++) {
        int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
        double dot = 0.0;
        for (int d = 0; d < ORC_DK; d++)
          dot += qd[d] * cached_value(kv, kv_dtype, slot, d, kv_scale);
        x[j - lo] = sm_scale * dot * LOG2E;
        if (x[j - lo] > m) m = x[j - lo];
      }
      double l = 0.0;
      for (int64_t j = lo; j < hi; j++) {
        int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
        double e = exp2(x[j - lo] - m);
        l += e;
        for (int d = 0; d < ORC_DV; d++)
          a[d] += e * cached_value(kv, kv_dtype, slot, d, kv_scale);
      }
      mx[base] = m;
      sm[base] = l;
      free(x);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Partials over caller-chosen token ranges.  The segmented decode keeps, per
 * segment, the local base-2 max, the exp2 sum and the unnormalised output of
 * the tokens in the segment's range [vLLM #51705, 实现拆解 4]; the pages cut
 * those ranges by the rule of oracle_segment_partials.  This function takes
 * the ranges as given, so that any partition of a request's tokens can be
 * checked slot by slot: row (t, h) of request b belongs to 64-row group
 * g = ((t - qo_indptr[b]) * H + h) / 64, and its slot s covers the tokens
 * [lo, hi) = ranges[((b * groups + g) * S + s) * 2 + {0, 1}] that the row
 * can see (j < row_len).  Per (row, head, slot), as oracle_segment_partials:
 *   m_s = max_j x_j, l_s = sum_j 2^(x_j - m_s), acc_s = sum_j 2^(x_j - m_s) vhat[j,:]
 * (-inf, 0, 0 for no visible token).  Output layout as there.               */
int oracle_range_partials(int num_reqs, int num_heads, int groups,
                          const int32_t *qo_indptr, const int32_t *row_len,
                          const uint16_t *q, const void *kv, int kv_dtype,
                          int64_t kv_rows, double kv_scale, double sm_scale,
                          const int32_t *block_table, int bt_stride,
                          int block_size, int num_slots, const int64_t *ranges,
                          double *acc, double *mx, double *sm) {
  const double LOG2E = 1.0 / log(2.0);
  int num_rows = qo_indptr[num_reqs];
  int S = num_slots;
  int err = ORC_OK;
  (void)kv_rows;
  if (S < 1 || groups < 1) return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < (int64_t)num_rows * num_heads; it++) {
    int row = (int)(it / num_heads);
    int h = (int)(it % num_heads);
    int b = request_of_row(num_reqs, qo_indptr, row);
    if (b < 0) {
#pragma omp atomic write
      err = ORC_ERR_ARG;
      continue;
    }
    int g = ((row - qo_indptr[b]) * num_heads + h) / 64;
    if (g >= groups) {
#pragma omp atomic write
      err = ORC_ERR_ARG;
      continue;
    }
    const uint16_t *qv = q + ((int64_t)row * num_heads + h) * ORC_DK;
    double qd[ORC_DK];
    for (int d = 0; d < ORC_DK; d++) qd[d] = bf16_bits_to_double(qv[d]);
    for (int s = 0; s < S; s++) {
      int64_t base = it * S + s;
      double *a = acc + base * ORC_DV;
      for (int d = 0; d < ORC_DV; d++) a[d] = 0.0;
      mx[base] = -INFINITY;
      sm[base] = 0.0;
      const int64_t *rg = ranges + (((int64_t)b * groups + g) * S + s) * 2;
      int64_t lo = rg[0] < 0 ? 0 : rg[0];
      int64_t hi = rg[1];
      if (hi > row_len[row]) hi = row_len[row];
      if (lo >= hi) continue;
      double *x = (double *)malloc(sizeof(double) * (size_t)(hi - lo));
      if (!x) {
#pragma omp atomic write
        err = ORC_ERR_NOMEM;
        break;
      }
      double m = -INFINITY;
      for (int64_t j = lo; j < hi; j++) {
        int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
        double dot = 0.0;
        for (int d = 0; d < ORC_DK; d++)
          dot += qd[d] * cached_value(kv, kv_dtype, slot, d, kv_scale);
        x[j - lo] = sm_scale * dot * LOG2E;
        if (x[j - lo] > m) m = x[j - lo];
      }
      double l = 0.0;
      for (int64_t j = lo; j < hi; j++) {
        int64_t slot = slot_of_token(block_table, bt_stride, b, j, block_size);
        double e = exp2(x[j - lo] - m);
        l += e;
        for (int d = 0; d < ORC_DV; d++)
          a[d] += e * cached_value(kv, kv_dtype, slot, d, kv_scale);
      }
      mx[base] = m;
      sm[base] = l;
      free(x);
    }
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Segment merge.  [vLLM #51705, 实现拆解 4 and the merge_mla_segments_triton
 * snippet]: base-2 segment statistics are combined into one output and a
 * natural-log LSE (the LOGE2 constant there is ln 2):
 *   M   = max_s m_s,   c_s = 2^(m_s - M)
 *   out = sum_s c_s acc_s / sum_s c_s l_s
 *   lse = (M + log2 sum_s c_s l_s) * ln 2
 * All segments empty (M = -inf): out = 0, lse = -inf.
 * Layout: acc [n_items, S, 512], m and l [n_items, S].                      */
void oracle_merge_segments(int64_t n_items, int num_segments, const double *acc,
                           const double *mx, const double *sm, double *out,
                           double *lse) {
  const double LN2 = log(2.0);
  int S = num_segments;
  for (int64_t it = 0; it < n_items; it++) {
    double M = -INFINITY;
    for (int s = 0; s < S; s++)
      if (mx[it * S + s] > M) M = mx[it * S + s];
    double *o = out + it * ORC_DV;
    for (int d = 0; d < ORC_DV; d++) o[d] = 0.0;
    if (M == -INFINITY) {
      lse[it] = -INFINITY;
      continue;
    }
    double denom = 0.0;
    for (int s = 0; s < S; s++) {
      double m_s = mx[it * S + s];
      if (m_s == -INFINITY) continue; /* an empty segment contributes nothing */
      double c = exp2(m_s - M);
      denom += c * sm[it * S + s];
      for (int d = 0; d < ORC_DV; d++)
        o[d] += c * acc[(it * S + s) * ORC_DV + d];
    }
    for (int d = 0; d < ORC_DV; d++) o[d] /= denom;
    lse[it] = (M + log2(denom)) * LN2;
  }
}

/* ------------------------------------------------------------------------ */
/* Cross-shard state merge in the natural-log domain.  [vLLM #51705, 功能与动机
 * and 实现拆解 4: rank-local partial outputs are merged through the DCP
 * attention merge, which consumes a natural-log LSE]; [sglang #34432, key
 * snippet: merge_state_triton(out_a, lse_a, out_b, lse_b)]:
 *   M   = max_r lse_r,   w_r = exp(lse_r - M)
 *   out = sum_r w_r out_r / sum_r w_r,   lse = M + ln sum_r w_r
 * A part with lse = -inf (an empty shard row) contributes nothing; all parts
 * empty gives out = 0, lse = -inf.
 * Layout: out_parts [W, n_items, 512], lse_parts [W, n_items].               */
void oracle_merge_states(int64_t n_items, int num_parts,
                         const double *out_parts, const double *lse_parts,
                         double *out, double *lse) {
  for (int64_t it = 0; it < n_items; it++) {
    double M = -INFINITY;
    for (int r = 0; r < num_parts; r++)
      if (lse_parts[r * n_items + it] > M) M = lse_parts[r * n_items + it];
    double *o = out + it * ORC_DV;
    for (int d = 0; d < ORC_DV; d++) o[d] = 0.0;
    if (M == -INFINITY) {
      lse[it] = -INFINITY;
      continue;
    }
    double denom = 0.0;
    for (int r = 0; r < num_parts; r++) {
      double l_r = lse_parts[r * n_items + it];
      if (l_r == -INFINITY) continue;
      double w = exp(l_r - M);
      denom += w;
      for (int d = 0; d < ORC_DV; d++)
        o[d] += w * out_parts[(r * n_items + it) * ORC_DV + d];
    }
    for (int d = 0; d < ORC_DV; d++) o[d] /= denom;
    lse[it] = M + log(denom);
  }
}

/* ------------------------------------------------------------------------ */
/* e4m3 ("fn") encoding of a float32 value, round to nearest even with
 * saturation to the largest finite magnitude 448 (NaN -> the NaN code 0x7F).
 * Written from the format's definition: every non-negative finite code
 * 0x00..0x7E is decoded with oracle_e4m3_to_double and the nearest one is
 * chosen; on an exact tie the code with an even mantissa (even code) wins.  */
uint8_t oracle_e4m3_encode_rne_sat(float xf) {
  double x = (double)xf;
  if (x != x) return 0x7F;
  uint8_t sign = 0;
  if (signbit(x)) { sign = 0x80; x = -x; }
  if (x >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double best_d = x;  /* distance to code 0 (value 0) */
  for (int c = 1; c <= 0x7E; c++) {
    double d = fabs(oracle_e4m3_to_double((uint8_t)c) - x);
    if (d < best_d || (d == best_d && (c % 2) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* Owner-filtered paged KV write.  [sglang #34432, 实现拆解 4 and the
 * forward_mla_rocm.py snippet: set_mla_kv_buffer writes the new tokens itself,
 * filtering by owner and dividing by the shard count; key snippet
 * g(j) = j * W + r].  Request b's qlen_b new tokens sit at global positions
 * g = L_b - qlen_b + t (t < qlen_b; row qo_indptr[b] + t of kv_new).  Rank
 * `rank` of W keeps the tokens it owns (g mod W == rank for interleave 1; the
 * generalisation above otherwise), at its local index j (g div W for
 * interleave 1), i.e. cache row block_table[b][j / block_size] * block_size +
 * j % block_size.  bf16 caches receive the row's 576 bf16 values unchanged;
 * fp8 caches receive e4m3 codes of (value / kv_scale) computed in float32
 * (round to nearest even, saturating).  Returns 0 or an error code.          */
int oracle_write_kv(int num_reqs, const int32_t *seq_lens, const int32_t *qo_indptr,
                    const uint16_t *kv_new, int world_size, int rank, int interleave,
                    const int32_t *block_table, int bt_stride, int block_size, void *cache,
                    int kv_dtype, float kv_scale, int64_t cache_rows) {
  if (world_size < 1 || rank < 0 || rank >= world_size || block_size < 1 || interleave < 1)
    return ORC_ERR_ARG;
  for (int b = 0; b < num_reqs; b++) {
    int qlen = qo_indptr[b + 1] - qo_indptr[b];
    int L = seq_lens[b];
    if (qlen < 1 || qlen > L) return ORC_ERR_QLEN;
    for (int t = 0; t < qlen; t++) {
      int64_t g = (int64_t)L - qlen + t;
      if (oracle_il_owner(g, world_size, interleave) != rank) continue;
      int64_t j = oracle_il_local_index(g, world_size, interleave);
      int32_t blk = block_table[(int64_t)b * bt_stride + j / block_size];
      int64_t slot = (int64_t)blk * block_size + j % block_size;
      if (blk < 0 || slot >= cache_rows) return ORC_ERR_SLOT;
      const uint16_t *src = kv_new + (int64_t)(qo_indptr[b] + t) * ORC_DK;
      for (int d = 0; d < ORC_DK; d++) {
        if (kv_dtype == 0) {
          ((uint16_t *)cache)[slot * ORC_DK + d] = src[d];
        } else {
          uint32_t u = ((uint32_t)src[d]) << 16;
          float v;
          memcpy(&v, &u, sizeof v);
          float q = v / kv_scale; /* float32 division, as the kernel does */
          ((uint8_t *)cache)[slot * ORC_DK + d] = oracle_e4m3_encode_rne_sat(q);
        }
      }
    }
  }
  return ORC_OK;
}
