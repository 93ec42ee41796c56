/*
 * mla_gb300.h -- C ABI of the GB300 (sm_103a) absorbed-form MLA decode /
 * causal multi-token speculative verify library (libmla_gb300.so).
 *
 * Pages cited (pull request digests):
 *   [vLLM #51705]   "ROCm AITER MLA supports causal multi-token speculative
 *                   verification under DCP"
 *   [sglang #34432] "[AMD][DCP 1/N] add dcp support for aiter backend"
 *   [vLLM #51011]   "fix silent wrong decoding of the fp8 KV cache on the ROCm
 *                   AITER MLA backend"
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except
 *     the argument structs themselves (host memory, read during the call) and
 *     mla_get_device_error's code_out (host).  The library never allocates or
 *     frees memory; the only scratch is the caller's workspace.
 *   - Every call is asynchronous on `stream` and performs no host
 *     synchronisation, except mla_get_device_error.  Grids are sized from the
 *     static bounds passed in, actual lengths are read on the device, so a
 *     sequence of calls can be captured in a CUDA graph and replayed with new
 *     lengths (the static-bound requirement of [vLLM #51705, 实现拆解 3]).
 *   - Arguments the host can check are checked before anything is launched;
 *     a failure returns a status and launches nothing.  Problems only the
 *     device can see (bad indices, lengths beyond a bound, a qlen that does
 *     not fit its seq_len) never fault: the kernel skips the bad access and
 *     records the first such problem in a device error word, read and cleared
 *     by mla_get_device_error.
 *   - Integers in device arrays are int32.  Row r of the flattened query /
 *     output view is (verify row t, head h) = (r / H, r % H).
 *
 * Tensor shapes (T = verify-row capacity, H = heads, B = requests):
 *   q        [T, H, 576] bf16: q_nope_out (512) then q_pe (64) per head
 *   kv_cache [N, 576] bf16, or [N, 576] fp8 e4m3 (OCP "fn") codes with one
 *            per-tensor float scale; a cached row is k_nope (512 latent, which
 *            is also V) then k_pe (64 rope)            [sglang #34432 snippet
 *            forward_mla_rocm.py: k = cat(k_nope, k_pe), v = k_nope]
 *   out      [T, H, 512] bf16;  lse [T, H] float32 natural log, heads unpadded
 *            [vLLM #51705, 实现拆解 4: unpadded LSE].
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t (struct CUstream_st *); 0 = legacy stream. */
typedef struct CUstream_st *mla_stream_t;

#define MLA_D_QK 576  /* q / K width: 512 latent + 64 rope   */
#define MLA_D_V 512   /* V / output width: the 512-d latent */
#define MLA_ABI_VERSION 5

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* a size, pointer or stride the host can see is wrong */
  MLA_ERR_UNSUPPORTED = 2,  /* valid but not supported: page size < 8, unknown dtype, ... */
  MLA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than mla_decode_verify_workspace() */
  MLA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed; see mla_last_error_string() */
  MLA_ERR_DEVICE_CHECK = 5  /* returned by mla_get_device_error when a device check fired */
} mla_status;

typedef enum mla_kv_dtype {
  MLA_KV_BF16 = 0,
  MLA_KV_FP8_E4M3 = 1
} mla_kv_dtype;

/* Device error codes (first one recorded wins; read with mla_get_device_error). */
typedef enum mla_device_error {
  MLA_DEV_OK = 0,
  MLA_DEV_BAD_INDPTR = 1,    /* qo_indptr not starting at 0, decreasing, or past the row capacity */
  MLA_DEV_BAD_QLEN = 2,      /* a request with qlen < 1 or qlen > seq_len */
  MLA_DEV_BAD_BLOCK_ID = 3,  /* a block-table entry needed for a visible token is < 0 or >= num_blocks */
  MLA_DEV_LEN_BOUND = 4,     /* a length exceeds the static bound (table width * page size) */
  MLA_DEV_BAD_SUBPAGE = 5,   /* the decode met a sub-page id outside the cache */
  MLA_DEV_WAIT_TIMEOUT = 6   /* an in-kernel wait gave up; the CTA returned without its result */
} mla_device_error;

/* Sub-page size P for a physical block size: the largest power of two dividing
 * block_size, capped at 128 [vLLM #51705, 实现拆解 3, _segmented_mla_page_size].
 * Returns -1 for block_size <= 0.  Host only, no CUDA call. */
int mla_page_size(int block_size);

/* Row plan [vLLM #51705, 实现拆解 2, _build_dcp_verify_row_view]: verify row t
 * of request b (qlen_b = qo_indptr[b+1] - qo_indptr[b] rows, seq_len L_b that
 * already counts the qlen_b new tokens) sees global positions
 * [0, L_b - qlen_b + t], so
 *     row_len[qo_indptr[b] + t] = L_b - qlen_b + 1 + t,  row_req[...] = b.
 * Rows in [qo_indptr[B], num_rows) get row_len 0 and row_req -1.
 * Optionally (block_table != NULL) it also expands the request's physical
 * block table into the sub-page table the decode reads [vLLM #51705, 实现拆解 3,
 * _fill_dcp_verify_page_table]: with P = mla_page_size(block_size) and
 * R = block_size / P,
 *     subpage_table[b][p] = block_table[b][p / R] * R + p % R  for p < cdiv(L_b, P),
 *     subpage_table[b][p] = -1                                 otherwise.
 * The cache is then addressed as rows id * P + offset of a [N, 576] view.
 * Rows of one request share one table row (they read the same KV).
 *   num_reqs B >= 0; num_rows T >= qo_indptr[B] (row-array capacity);
 *   seq_lens [B]; qo_indptr [B+1]; row_len, row_req [T] outputs;
 *   block_table [B, block_table_stride] (entries for blocks a request does
 *   not use are ignored), num_blocks bounds its entries; subpage_table
 *   [B, subpage_stride] output; subpage_stride * P is the static length bound.
 * Device checks: MLA_DEV_BAD_INDPTR, MLA_DEV_BAD_QLEN (the row lengths of that
 * request are then written as 0), MLA_DEV_BAD_BLOCK_ID (entry -1), and
 * MLA_DEV_LEN_BOUND (L_b > subpage_stride * P; the table row is truncated). */
mla_status mla_plan_rows(int num_reqs, int num_rows, const int32_t *seq_lens,
                         const int32_t *qo_indptr, int32_t *row_len,
                         int32_t *row_req, const int32_t *block_table,
                         int block_table_stride, int num_blocks,
                         int block_size, int32_t *subpage_table,
                         int subpage_stride, mla_stream_t stream);

/* Shard row view for rank `rank` of `world_size` round-robin context shards
 * [vLLM #51705, 实现拆解 2 and the _build_dcp_verify_row_view snippet;
 * sglang #34432, key snippet g(j) = j * W + r]: global position g lives on
 * rank g mod W at local index g div W, so a row whose global window holds w
 * positions sees
 *     row_len_local = floor((w - 1 - rank) / W) + 1  if w - 1 - rank >= 0, else 0
 * tokens of this rank -- counted from the row's own global window, never as
 * "request's local length minus the causal offset".  interleave I > 1 goes
 * beyond the pages, which accept only I = 1 [vLLM #51705, 实现拆解 1,
 * _segmented_dcp_verify_supported]: runs of I consecutive positions are
 * dealt to the ranks in turn, position g on rank (g div I) mod W at local
 * index (g div (I*W)) * I + g mod I, and the rank sees
 *     row_len_local = (w div (I*W)) * I + clamp(w mod (I*W) - rank * I, 0, I).
 * interleave < 1 returns MLA_ERR_INVALID_ARG.
 * Optionally (block_table != NULL, the SHARD's own physical block table over
 * its local tokens) it writes the shard's sub-page table exactly as
 * mla_plan_rows does, sized by the request's longest shard-local row; the
 * static bound (sglang #34432: ceil(max_context / W)) is
 * subpage_stride * P.  Device checks as mla_plan_rows. */
mla_status mla_shard_row_view(int num_reqs, int num_rows,
                              const int32_t *qo_indptr,
                              const int32_t *row_len_global, int world_size,
                              int rank, int interleave, int32_t *row_len_local,
                              const int32_t *block_table,
                              int block_table_stride, int num_blocks,
                              int block_size, int32_t *subpage_table,
                              int subpage_stride, mla_stream_t stream);

/* All world_size shard row views of one step in one launch -- the ranks of a
 * context-sharded step simulated on one GPU (the pages run one view per
 * rank).  View r is exactly mla_shard_row_view(rank = r): it reads
 * block_tables + r * num_reqs * block_table_stride (rank r's own table over
 * its local tokens, when block_tables != NULL) and writes
 * row_len_local + r * num_rows and subpage_tables + r * num_reqs *
 * subpage_stride, i.e. row_len_local [W, T] and subpage_tables [W, B, stride]
 * as mla_decode_verify's num_views = W reads them.  1 <= world_size <= 65535;
 * errors and device checks as mla_shard_row_view. */
mla_status mla_shard_row_views(int num_reqs, int num_rows,
                               const int32_t *qo_indptr,
                               const int32_t *row_len_global, int world_size,
                               int interleave, int32_t *row_len_local,
                               const int32_t *block_tables,
                               int block_table_stride, int num_blocks,
                               int block_size, int32_t *subpage_tables,
                               int subpage_stride, mla_stream_t stream);

/* Arguments of mla_decode_verify (host struct, read during the call). */
typedef struct mla_decode_args {
  int num_reqs;          /* B >= 1 */
  int num_rows;          /* T: row capacity of q / out / lse; qo_indptr[B] <= T */
  int num_heads;         /* H >= 1, unpadded */
  int max_qlen;          /* static bound on qlen_b (sizes the grid) */
  int kv_dtype;          /* mla_kv_dtype */
  float sm_scale;        /* softmax scale applied to the full 576-d dot product */
  float kv_scale;        /* per-tensor dequant scale (fp8); ignored for bf16 */
  const void *q;         /* [T, H, 576] bf16 */
  const void *kv_cache;  /* [num_cache_rows, 576] bf16 or e4m3; 16-byte aligned */
  int64_t num_cache_rows;
  const int32_t *qo_indptr;      /* [B+1] */
  const int32_t *row_len;        /* [T] tokens row r sees, in this cache's index space */
  const int32_t *subpage_table;  /* [B, subpage_stride] sub-page ids (mla_plan_rows) */
  int subpage_stride;
  int page_size;         /* P = mla_page_size(block_size); 8 <= P <= 128 */
  int num_segments;      /* S: split-K segment slots per (view, request, row
                          * block), 1 <= S <= 1024 -- see mla_decode_flags */
  void *out;             /* [T, H, 512] bf16 output */
  float *lse;            /* [T, H] natural-log LSE (-inf for a row with no tokens) */
  int flags;             /* bitwise OR of mla_decode_flags (0 = default) */
  /* V row views of the same queries in one call (0 or 1 = one view): view v
   * reads row_len[v*T + r] and subpage_table[(v*B + b) * subpage_stride + p]
   * and writes out[(v*T + r), h] / lse[(v*T + r), h] -- e.g. the W shard row
   * views of one batch, whose outputs form the [W, T, H] shard states of the
   * state merge.  row_len is [V, T], subpage_table [V, B, stride], out
   * [V, T, H, 512], lse [V, T, H]; no counterpart in the pages, which run one
   * decode per rank. */
  int num_views;
  /* Bound on every in-kernel wait for the work to progress, in SM clock
   * cycles; 0 = the default of 4e9 cycles (about 2 s).  A wait that runs out
   * records MLA_DEV_WAIT_TIMEOUT and the kernel returns without its result
   * (it first lets its own copies and MMAs in flight finish, under a separate
   * fixed bound).  Only a caller that wants to exercise that exit path needs
   * a small value. */
  int64_t wait_cycles;
} mla_decode_args;

typedef enum mla_decode_flags {
  /* With num_segments > 1: launch only the decode kernel, leaving the segment
   * partials in the workspace (layout of mla_decode_verify_workspace) for the
   * caller's own mla_merge_segments call; out / lse are not written.  This is
   * the pages' two-step form (segmented decode, then merge_mla_segments). */
  MLA_DECODE_SKIP_MERGE = 1,
  /* How the S > 1 segment slots are filled.  Default (flag clear, at most
   * 1024 (view, request, row block) units, and units x the static bound's
   * tiles plus one (subpage_stride * P / 64 + 1) within int32): balanced
   * split -- every unit with tiles counts as one overhead position (its Q load
   * and epilogue cost about one tile) followed by its 64-token KV tiles; the
   * positions of all units, laid end to end in unit order, are cut into
   * equal contiguous chunks, one per SM (grown where needed so that no unit
   * meets more than S chunks); the part of a unit inside chunk c is its
   * segment c - c0 (c0: the first chunk holding one of its tiles), and slots
   * past a unit's last part hold max = -inf, sum = 0.  Every SM then does
   * the same work, whatever the mix of lengths.  With this flag (or beyond those
   * bounds): the pages' split [vLLM #51705, 实现拆解 4] -- segment s of a request holds
   * tokens [s*L, (s+1)*L) with L = ceil(len / (S*P)) * P, len the
   * request's longest visible row.  The merged out / lse are the same either
   * way up to float rounding. */
  MLA_DECODE_UNIFORM_SEGMENTS = 2,
  /* With the balanced split: merge the split-K parts inside the decode kernel
   * instead of a separate merge launch.  A unit lying inside one SM's chunk
   * is written as bf16 out + LSE straight from its accumulator; the parts of
   * a unit cut across chunks are published to the workspace (a release add
   * on a per-unit counter), and the SMs holding them merge its 64-dim output
   * blocks once their own tiles are done (a holder waits, bounded, only when
   * every chunk of the unit is claimed by a running SM; the last part to
   * arrive merges whatever no holder claimed).  The result is the same up to
   * float rounding.  Needs num_segments > 1 and neither flag above
   * (MLA_ERR_UNSUPPORTED otherwise, or when the call cannot take the
   * balanced split).  Off by default: on this library's configured workloads
   * the merge tail inside the kernel measured slower than the separate merge. */
  MLA_DECODE_FUSED_MERGE = 4
} mla_decode_flags;

/* Workspace bytes mla_decode_verify needs for `a`.  Layout, each region
 * starting on a 256-byte boundary, in this order:
 *   segm_out [V, B, RB, S, 8, 512, 8] bf16: RB = ceil(max_qlen * H / 64) row
 *     blocks per request; block (v, b, rb, s) holds segment s of view v's
 *     rows rb*64 .. rb*64 + 63 of request b (a request's rows numbered
 *     t * H + h) as [row octet][dim][row within the octet]: block row i, dim d
 *     at ((i / 8) * 512 + d) * 8 + i % 8; rows past qlen * H are unused;
 *   segm_max [V, T, H, S] float32, segm_sum [V, T, H, S] float32
 *   (these three only when num_segments > 1), then 256 bytes of scheduler
 *   state (a work counter the call zeroes on the stream before its kernel).
 * Host only. */
size_t mla_decode_verify_workspace(const mla_decode_args *a);

/* Absorbed-form MLA decode / causal verify over the paged latent cache.
 * For each row r (request b) and head h, with n_r = row_len[r] visible tokens
 * j = 0 .. n_r - 1 of request b (token j is cache row
 * subpage_table[b][j / P] * P + j % P):
 *   s_j = sm_scale * <q[r,h,:], k_j>   over all 576 dims (fp8: k_j = kv_scale * code)
 *   out[r,h,:] = sum_j softmax(s)_j * k_j[0:512],  lse[r,h] = ln sum_j e^{s_j}
 * [sglang #34432 snippets; vLLM #51705, 实现拆解 2].  Rows of a request are
 * processed jointly against shared KV tiles with per-row causal masks; the
 * rows' lengths may differ by any amount.  With num_segments S > 1 the KV
 * tokens of each (view, request, 64-row block) are split into up to S
 * segment slots -- by default the balanced split, with
 * MLA_DECODE_UNIFORM_SEGMENTS the pages' equal split (see mla_decode_flags)
 * -- whose base-2 partials (max, exp2-sum, unnormalised output) go to the
 * workspace and are merged into bf16 out + natural-log LSE by the segment
 * merge [vLLM #51705, 实现拆解 4]; S == 1 writes out/lse directly.
 * fp8 codes are converted to bf16 exactly; kv_scale is folded into the score
 * scale and into the output.  The query-by-key products use bf16 tensor-core
 * MMAs with float32 accumulation; softmax probabilities are rounded to bf16
 * for the PV product.
 * Returns MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED / MLA_ERR_WORKSPACE before
 * launching anything; MLA_ERR_CUDA if a launch fails.  Device checks:
 * MLA_DEV_LEN_BOUND (row_len > subpage_stride * P: the row is clipped),
 * MLA_DEV_BAD_SUBPAGE (id outside the cache: the page is read as zeros),
 * MLA_DEV_WAIT_TIMEOUT. */
mla_status mla_decode_verify(const mla_decode_args *a, void *workspace,
                             size_t workspace_bytes, mla_stream_t stream);

typedef enum mla_merge_mode {
  MLA_MERGE_SEGMENTS = 0, /* base-2 segment partials of one rank */
  MLA_MERGE_STATES = 1    /* natural-log (out, lse) states of W shards */
} mla_merge_mode;

/* Arguments of mla_merge_segments (host struct, read during the call). */
typedef struct mla_merge_args {
  int mode;        /* mla_merge_mode */
  int num_rows;    /* T */
  int num_heads;   /* H */
  int num_parts;   /* S segments or W shards, 1 <= num_parts <= 1024 */
  /* MLA_MERGE_SEGMENTS: the decode workspace's partials: segm_out
   * [B, RB, S, 8, 512, 8] bf16 unnormalised outputs (uint16 bit patterns; the
   * block layout of mla_decode_verify_workspace), segm_max / segm_sum
   * [T, H, S] float32 base-2 maxima and exp2 sums.  A part with max = -inf
   * is empty and contributes nothing (its output is not read as a value). */
  const uint16_t *segm_out;
  const float *segm_max;
  const float *segm_sum;
  const int32_t *qo_indptr;  /* segment mode: [B + 1] device, as for mla_decode_verify */
  int num_reqs;              /* segment mode: B */
  int max_qlen;              /* segment mode: bound on qlen_b, fixes RB */
  int num_views;             /* segment mode: V row views (0 or 1 = one); out / lse are
                              * then [V, T, H, 512] / [V, T, H], the partials as above */
  /* MLA_MERGE_STATES: [W, T, H, 512] bf16 outputs and [W, T, H] float32
   * natural-log LSEs; a part with lse = -inf is empty and never read. */
  const void *part_out;
  const float *part_lse;
  void *out;       /* [T, H, 512] bf16 */
  float *lse;      /* [T, H] float32 natural log */
} mla_merge_args;

/* Merge of partial attention states.
 * Segment mode [vLLM #51705, 实现拆解 4, merge_mla_segments_triton]:
 *   M = max_s m_s, c_s = 2^(m_s - M), out = sum_s c_s acc_s / sum_s c_s l_s,
 *   lse = (M + log2 sum_s c_s l_s) * ln 2.
 * State mode [vLLM #51705, 功能与动机: rank partials merged by the DCP merge;
 * sglang #34432, merge_state_triton and 评论区精华 4 (base e)]:
 *   M = max_r lse_r, w_r = e^(lse_r - M), out = sum_r w_r out_r / sum_r w_r,
 *   lse = M + ln sum_r w_r.
 * All parts empty: out = 0, lse = -inf.  out is rounded to bf16 (RNE). */
mla_status mla_merge_segments(const mla_merge_args *a, mla_stream_t stream);

/* Owner-filtered paged write of the new verify tokens -- the step right before
 * the decode [sglang #34432, 实现拆解 4 and forward_mla_rocm.py snippet:
 * set_mla_kv_buffer filters by owner and divides by the shard count; key
 * snippet g(j) = j * W + r].  Request b's qlen_b new tokens (rows
 * qo_indptr[b] .. qo_indptr[b+1]-1 of kv_new, each [576] bf16 = k_nope then
 * k_pe) sit at global positions g = L_b - qlen_b + t.  Rank `rank` of
 * `world_size` keeps the tokens with g mod W == rank, at its local index
 * j = g div W: cache row block_table[b][j / block_size] * block_size +
 * j % block_size of this rank's cache [num_cache_rows, 576].  world_size = 1
 * is the plain (unsharded) write.  bf16 caches receive the values unchanged;
 * fp8 caches (kv_dtype = MLA_KV_FP8_E4M3) receive the e4m3 codes of
 * value / kv_scale computed in float32, rounded to nearest even and
 * saturated to +-448.  interleave I > 1 places position g on rank
 * (g div I) mod W at local index (g div (I*W)) * I + g mod I, as
 * mla_shard_row_view counts it.
 * Device checks: MLA_DEV_BAD_INDPTR, MLA_DEV_BAD_QLEN, MLA_DEV_BAD_BLOCK_ID
 * (the token is then not written). */
mla_status mla_write_kv(int num_reqs, int num_rows, const int32_t *seq_lens,
                        const int32_t *qo_indptr, const void *kv_new, int world_size,
                        int rank, int interleave, const int32_t *block_table,
                        int block_table_stride, int num_blocks, int block_size,
                        void *kv_cache, int kv_dtype, float kv_scale,
                        int64_t num_cache_rows, mla_stream_t stream);

/* The same decode / verify as mla_decode_verify, for callers that cannot
 * allocate device memory where they make the call -- serving runtimes that
 * reserve all device memory at start-up and forbid allocation on the request
 * path, and plain C or plugin hosts that hold no device allocator (for them a
 * cudaMalloc would also synchronise the device mid-step).  The pages have no
 * counterpart: this is a deployment convenience of this library.
 * The scratch mla_decode_verify would take from the caller's workspace is
 * instead a fixed array of MLA_STATIC_SCRATCH_BYTES in the library's device
 * memory, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing (no cudaMalloc / cudaFree, no allocating
 * library routine).  Problems whose mla_decode_verify_workspace(a) exceeds the
 * array are rejected with MLA_ERR_WORKSPACE before anything is launched.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array per device and leaves its
 * contents behind (the work counter in it is zeroed on the stream by each
 * call): calls whose work overlaps on the GPU -- on different streams, or from
 * different host threads -- race on it and must be serialised by the caller.
 * Arguments, outputs and errors are otherwise those of mla_decode_verify. */
#define MLA_STATIC_SCRATCH_BYTES (80u * 1024u * 1024u)
mla_status mla_decode_verify_noalloc(const mla_decode_args *a, mla_stream_t stream);

/* Synchronises `stream`, returns the first device error code recorded on the
 * current device since the last call (MLA_DEV_OK if none) in *code_out, and
 * clears it.  Returns MLA_ERR_DEVICE_CHECK if a code was recorded, MLA_OK if
 * not, MLA_ERR_CUDA if the synchronisation failed. */
mla_status mla_get_device_error(int32_t *code_out, mla_stream_t stream);

/* Text of the last host-side error of the calling thread ("" if none). */
const char *mla_last_error_string(void);

/* Name of a status code. */
const char *mla_status_string(int status);

/* MLA_ABI_VERSION of the loaded library. */
int mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
