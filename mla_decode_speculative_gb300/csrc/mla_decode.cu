// mla_decode.cu -- absorbed-form MLA decode / causal multi-token verify over a
// paged latent KV cache.
//
// What it computes (sglang #34432 digest, forward_mla_rocm.py snippet;
// vLLM #51705 digest, 实现拆解 2-4): for every query row r = (verify row t,
// head h) of request b and every visible token j < row_len[t],
//   s_j = sm_scale * kv_scale * <q[r, 0:576], k_j[0:576]>,  v_j = k_j[0:512],
// with an online (base-2) softmax over the tokens of one split-K segment; the
// segment's (max, exp2-sum, unnormalised output) partial is written for the
// segment merge, or, with a single segment, the normalised bf16 output and
// natural-log LSE directly.
//
// GB300 design (not the pages' ROCm design):
//  * Work entry = (row view, request, block of <= 64 query rows, split-K
//    segment slot, token range).  The rows of a request (heads x qlen) are
//    decoded jointly against shared 64-token KV tiles, so each latent row is
//    read from HBM once per request (the pages replicate the request once per
//    verify row); several row views of the same queries (the shard views of a
//    DCP step) can share one launch.
//  * Persistent CTAs, one per SM.  Balanced split (default): every CTA
//    tabulates the tiles of all (view, request, row block) units, counts one
//    overhead position per unit with tiles (a part's Q load and epilogue),
//    and CTA c takes chunk c of the concatenated positions (the in-kernel
//    merge variant claims chunks from an atomic counter); a chunk's part of
//    each unit whose tiles it meets is one segment of that unit.  With the
//    pages' equal split the producer claims (unit, segment) items from an
//    atomic counter, longest requests first.  Entries, with their rows'
//    visible lengths, go to the other roles through a 4-deep shared-memory
//    work ring.  Every barrier phase follows one running tile counter.
//  * Swapped operand order, so the output accumulator fits TMEM densely:
//        S^T[64 tok, 64 rows]     = K_tile[64, 576] . Q[64, 576]^T      (M = 64, K-major A and B)
//        O^T[4x128 dims, 64 rows] += V^T[512, 64 tok] . P^T[64, 64]^T   (M = 128, MN-major A and B)
//    TMEM: O^T in columns 0-255 (4 blocks x 64), S^T of stage s in columns
//    256 + 64 s (an M = 64 result puts token 16 q + i in lane 32 q + i).
//  * Two shared-memory stages of one 64-token tile each: nine 8 KB chunks of
//    64 tokens x 64 dims (128-byte swizzle; one 3-D TMA box per tile when the
//    page size is >= 64), the eight V chunks adjacent so PV reads them in
//    place, the rope chunk last; once QK has retired a stage's rope chunk it
//    receives that tile's P^T.  Q (64 x 576) is resident per item.
//  * The UMMA warp runs an event loop over non-blocking barrier tests: a PV
//    whose P^T is ready goes first (it frees a stage for the next load), QK of
//    the next tile runs while the softmax of the current one is under way.
//  * Warp roles: warps 0-7 softmax (column group g = warp / 4 owns rows
//    32g..32g+31; TMEM lane quarter = warp % 4), warp 8 TMA producer, warp 9
//    UMMA issuer and TMEM owner.  fp8 tiles are TMA-loaded packed into the
//    stage's upper half and expanded in place to bf16 by the softmax warps.
//  * Lazy rescaling: the running reference max only moves when a tile's max
//    exceeds it by more than 2^8, so O is rarely rescaled in TMEM.
//  * Every wait is bounded; a timeout records MLA_DEV_WAIT_TIMEOUT, lets all
//    roles drain without skipping a barrier, frees TMEM and returns.
//  * Launched with programmatic stream serialization: barriers and TMEM are
//    set up while the previous kernel in the stream finishes, and nothing
//    touches global memory before griddepcontrol.wait.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {
namespace {

constexpr int kTileTok = 64;       // KV tokens per tile (UMMA M of the QK product)
constexpr int kRows = 64;          // query rows per work item (UMMA N)
constexpr int kNumChunks = 9;      // 576 / 64 dims per 128-byte swizzled chunk
constexpr int kStages = 2;         // tiles in flight
constexpr int kPChunk = 8;         // rope chunk of a stage, then the tile's P^T
constexpr int kChunkBytes = kTileTok * 128;            // 8 KB
constexpr int kStageBytes = kNumChunks * kChunkBytes;  // 72 KB
constexpr int kQChunkBytes = kRows * 128;              // 8 KB
constexpr int kNumSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;   // stage s: + 64 s
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr long long kPvGrace = 1200;           // SM cycles a ready QK waits for a pending P^T
constexpr long long kPvGraceLast = 20000;      // ... when that P^T is an item's last (its epilogue waits)
constexpr float kLn2 = 0.69314718055994530942f;

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kStageBytes;
constexpr int kOffMisc = kOffQ + kNumChunks * kQChunkBytes;

// One claimed work item as published by the producer to the other roles.
struct WorkEntry {
  int w;          // claim index (item or chunk), -1 = no more work
  int b, rb, seg, q_row, row_base, n_rows, seg_lo, seg_hi, n_tiles;  // b: view * B + request
  int fill_hi;    // segment slots seg+1 .. fill_hi-1 of these rows get no part: mark them empty
  int unit;       // balanced split: the (view, request, row block) unit of this part
  int n_parts;    // balanced split: parts the unit has (0: a unit without tiles)
  int c_last;     // balanced split: chunk holding the unit's last part
  alignas(16) int lens[kRows];  // visible tokens of each of the block's rows (0 past n_rows)
};
constexpr int kWorkRing = 4;
constexpr int kMaxOrderedReqs = 128;  // requests ranked longest-first in every CTA
constexpr int kMaxUnits = 1024;       // balanced split: (view, request, row block) units tabulated per CTA

// In-kernel split-K merge (balanced split): a part of a multi-part unit that
// this CTA computed; it is published, and the unit's claimed 64-dim output
// blocks merged, once the CTA's own work is done.
struct PendMerge {
  int b, rb, row_base, n_rows, n_parts, unit;
  int seg, c_last;  // this part's index in the unit; chunk of the unit's last part
  unsigned todo;    // bit k: output dims 64k .. 64k + 63 are merged by this CTA
  int wait;         // 1: wait until every part of the unit is published
  int go;           // the unit is complete (or this CTA's wait ran out: 0)
  int staged;       // byte offset of its parts' slices in the staging area, -1: read from L2 directly
};
constexpr int kMaxPend = 4;  // one chunk per CTA holds at most two multi-part units

struct Misc {
  uint64_t full[kStages];
  uint64_t ready[kStages];    // fp8 only: stage expanded to bf16
  uint64_t empty[kStages];
  uint64_t s_full[kStages];   // QK of the stage's tile retired
  uint64_t p_full[kStages];   // P^T of the stage's tile written
  uint64_t o_done[kStages];   // PV of the stage's tile retired
  uint64_t q_full, q_empty, fin;
  uint64_t work_full[kWorkRing], work_empty[kWorkRing];
  uint32_t tmem_base;
  int abort;
  WorkEntry work[kWorkRing];
  int sm_stop[2];  // softmax warps' shared exit decision (double-buffered)
  int req_key[kMaxOrderedReqs];   // a request's longest row (producer's scratch)
  int req_order[kMaxOrderedReqs]; // requests, longest first
  int unit_end[kMaxUnits];        // balanced split: tiles of unit u, then positions of units 0..u (prefix sum)
  float red[2][2][4][32];  // [buffer][column group][lane quarter][lane]
  PendMerge pend[kMaxPend];       // softmax warps: merges to run after the CTA's own parts
  int n_pend;
  int merge_go;
};
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc)) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kStageBytes % 1024 == 0 && kOffQ % 1024 == 0, "swizzle-atom alignment");

struct Params {
  const int32_t *qo_indptr;
  const int32_t *row_len;
  const int32_t *subpage_table;
  __nv_bfloat16 *segm_out;  // unnormalised partial outputs, bf16
  float *segm_max;
  float *segm_sum;
  __nv_bfloat16 *out;
  float *lse;
  int *err;
  int *sched;              // work-claim counter, zero at launch
  unsigned *unit_state;    // per unit: parts published (bits 0-15), output blocks claimed by waiting holders (16-23)
  int64_t num_cache_rows;
  long long wait_budget;   // SM cycles any wait on the work may take before the CTA gives up
  long long drain_budget;  // SM cycles the exit path waits for this CTA's own copies and MMAs
  int subpage_stride;
  int page_size;
  int num_heads;
  int num_segments;
  int row_blocks;
  int num_items;           // num_reqs * num_views * row_blocks * num_segments
  int num_reqs;
  int num_views;           // row views of the same queries decoded in one launch
  int max_qlen;
  int num_rows;
  int max_len;
  int tile3d;              // KV tensor map is the 3-D whole-tile view (page size >= 64)
  int balanced;            // split-K by equal chunks of the units' positions (else S equal segments per request)
  int fused;               // balanced split merged in this kernel into out / lse (no merge launch)
  int num_units;           // num_views * num_reqs * row_blocks
  float score_scale_log2;  // sm_scale * kv_scale * log2(e)
  float out_scale;         // kv_scale (fp8) or 1
};

__device__ __forceinline__ void record_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Fills the request / row-block part of a work entry (the whole producer
// warp): rows of the block and the visible length of each, and returns the
// request's longest visible length (every row clamped to [0, max_len]) in
// group_len.  Returns false when the request's qo_indptr is inconsistent (the
// entry then has no rows).  Requests with more than 32 verify rows read the
// extra lengths directly.
__device__ __forceinline__ bool decode_unit(const Params &p, int v, int b, int rb, WorkEntry &e, int lane,
                                            bool &clipped, int &group_len) {
  const int vrow = v * p.num_rows;  // view v's rows start here in row_len / out / lse
  const int q0 = p.qo_indptr[b];
  const int q1 = p.qo_indptr[b + 1];
  clipped = false;
  bool ok = !(q0 < 0 || q1 < q0 || q1 > p.num_rows || q1 - q0 > p.max_qlen);
  const int qlen = ok ? q1 - q0 : 0;
  const int rows_req = qlen * p.num_heads;
  const int row_begin = rb * kRows;
  const int n_rows = row_begin < rows_req ? min(kRows, rows_req - row_begin) : 0;
  // lengths of the request's rows: lane t holds row t (t < 32)
  int my_len = 0;
  if (lane < qlen) my_len = p.row_len[vrow + q0 + lane];
  group_len = 0;
  for (int t = lane; t < qlen; t += 32) {
    int l = t == lane ? my_len : p.row_len[vrow + q0 + t];
    if (l > p.max_len) { clipped = true; l = p.max_len; }
    group_len = max(group_len, max(l, 0));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) group_len = max(group_len, __shfl_xor_sync(0xffffffffu, group_len, o));
  clipped = __any_sync(0xffffffffu, clipped);
  // per-column lengths: column c is row (row_begin + c) / H of the request
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    const int t = (row_begin + c) / p.num_heads;
    const int tt = t < 32 ? t : 0;
    int l = __shfl_sync(0xffffffffu, my_len, tt);
    if (t >= 32 && c < n_rows) l = p.row_len[vrow + q0 + t];
    e.lens[c] = c < n_rows ? min(max(l, 0), p.max_len) : 0;
  }
  if (lane == 0) {
    e.b = v * p.num_reqs + b;
    e.rb = rb;
    e.q_row = q0 * p.num_heads + row_begin;
    e.n_rows = n_rows;
    e.row_base = (vrow + q0) * p.num_heads + row_begin;
  }
  return ok;
}

// The same longest visible length, by one thread (the balanced split's unit
// table); 0 for an inconsistent qo_indptr.
__device__ __forceinline__ int request_len(const Params &p, int v, int b) {
  const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.num_rows || q1 - q0 > p.max_qlen) return 0;
  const int32_t *rl = p.row_len + static_cast<int64_t>(v) * p.num_rows;
  int len = 0;
  for (int t0 = q0; t0 < q1; t0 += 8) {  // eight loads in flight, then the max
    int l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) l[k] = t0 + k < q1 ? rl[t0 + k] : 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) len = max(len, min(max(l[k], 0), p.max_len));
  }
  return len;
}

// Warp transpose-reduce: on entry v[k] is this lane's value of column k; on
// exit v[0] holds the max (or sum) over the 32 lanes of column `lane`.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = upper ? v[k] : v[k + off];
      const float keep = upper ? v[k + off] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// Half-warp transpose-reduce: lanes 16h .. 16h + 15 each hold 16 values
// (column 16h + k in v[k]); on exit lane L holds the max (or sum) over its
// half's 16 lanes of column L.
template <bool kMax>
__device__ __forceinline__ float half_reduce_scatter(float (&v)[16], int lane) {
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = upper ? v[k] : v[k + off];
      const float keep = upper ? v[k + off] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr)
               : "memory");
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
// Two e4m3 codes (low byte first) -> two bf16 (exact; NaN stays NaN).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
  return pack_bf16(f.x, f.y);
}

// ---- in-kernel split-K merge (balanced split)

__device__ __forceinline__ int ld_volatile(const int *ptr) {
  int v;
  asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *ptr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_release_gpu(unsigned *ptr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}

constexpr uint32_t kMergeBar = 5;                        // named barrier of the 256 softmax threads
constexpr int kMergeThreads = kNumSoftmaxWarps * 32;
constexpr int kMergeSlots = 32;                          // parts whose weights are staged at a time

// Shared-memory scratch of one block merge (inside stage 0, free once the
// CTA's own tiles are done).
constexpr int kMergePassDims = 128;                     // output dims merged per pass
struct MergeScratch {
  float m[kMergeSlots][kRows];         // base-2 max of (part, row), parts 0 .. 31
  float w[kMergeSlots][kRows];         // normalised weight of (part, row), 32 parts at a time
  uint16_t o[kRows][kMergePassDims + 8];  // merged bf16 [row][dim] of one pass, padded rows
  float M[kRows], inv[kRows];          // row max (base 2) and 1 / denominator
  float part_m[4][kRows], part_d[4][kRows];
};
static_assert(sizeof(MergeScratch) <= kStageBytes, "merge scratch fits one stage");

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *gptr) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kStagingBytes = kStages * kStageBytes;  // the two stages, free once the CTA's tiles are done

// The claimed output dims of a unit as one run of consecutive 64-dim blocks:
// (first block, number of blocks), or nb = 0 when the claim is not one run.
__device__ __forceinline__ void todo_run(unsigned todo, int &b0, int &nb) {
  b0 = __ffs(todo) - 1;
  nb = __popc(todo);
  if (((todo >> b0) & ((1u << nb) - 1u)) != ((1u << nb) - 1u)) nb = 0;
}

// Issues the copies of a staged unit's parts into shared memory: for every
// part u and row octet o, the claimed dims' 16-byte (8-row) pieces, as
// [part][octet][dim] (cp.async, 16 bytes per thread and instruction; a warp
// covers 512 consecutive bytes).
__device__ void stage_unit(const Params &p, const PendMerge &pm, uint32_t s_stage, int tid) {
  int b0, nb;
  todo_run(pm.todo, b0, nb);
  const int D = 64 * nb, S = p.num_segments;
  const int64_t blk0 = (static_cast<int64_t>(pm.b) * p.row_blocks + pm.rb) * S;
  const int total = pm.n_parts * 8 * D;
  const uint32_t dst0 = s_stage + static_cast<uint32_t>(pm.staged);
  for (int c = tid; c < total; c += kMergeThreads) {
    const int d = c % D, uo = c / D;  // uo = part * 8 + octet
    const int u = uo >> 3, o = uo & 7;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.segm_out + (blk0 + u) * (512 * kRows)) + o * 512 + 64 * b0 + d;
    cp_async16(dst0 + static_cast<uint32_t>(c) * 16u, src);
  }
}

// Per-row max and denominator of a unit's n published parts, and the
// natural-log LSE (written when write_lse): four threads per row, parts
// strided by 4, a running (max, sum) rescaled as the max grows; the maxima of
// the first 32 parts stay in shared memory for the weights.
__device__ void merge_unit_stats(const Params &p, const PendMerge &pm, bool write_lse, int tid, MergeScratch &ms) {
  const int S = p.num_segments, n = pm.n_parts;
  const float *mx = p.segm_max + static_cast<int64_t>(pm.row_base) * S;  // [rows][S]
  const float *sm = p.segm_sum + static_cast<int64_t>(pm.row_base) * S;
  const int row = tid & (kRows - 1), quarter = tid >> 6;
  float Mq = -INFINITY, dq = 0.0f;
  auto take = [&](float m, float l) {
    if (m == -INFINITY) return;
    if (m > Mq) {
      dq = dq * exp2f(Mq - m) + l;  // 0 while Mq is -inf
      Mq = m;
    } else {
      dq += exp2f(m - Mq) * l;
    }
  };
  {
    float mv[8], lv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int s2 = quarter + 4 * j;
      const bool in = row < pm.n_rows && s2 < n;
      mv[j] = in ? __ldcg(mx + row * S + s2) : -INFINITY;
      lv[j] = in ? __ldcg(sm + row * S + s2) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      take(mv[j], lv[j]);
      ms.m[quarter + 4 * j][row] = mv[j];
    }
  }
  if (row < pm.n_rows)
    for (int s2 = quarter + 4 * 8; s2 < n; s2 += 4) take(__ldcg(mx + row * S + s2), __ldcg(sm + row * S + s2));
  ms.part_m[quarter][row] = Mq;
  ms.part_d[quarter][row] = dq;
  named_bar_sync(kMergeBar, kMergeThreads);
  if (quarter == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) M = fmaxf(M, ms.part_m[k][row]);
    float d = 0.0f;
    if (M != -INFINITY)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (ms.part_m[k][row] != -INFINITY) d += exp2f(ms.part_m[k][row] - M) * ms.part_d[k][row];
    ms.M[row] = M;
    ms.inv[row] = d > 0.0f ? 1.0f / d : 0.0f;
    if (write_lse && row < pm.n_rows) p.lse[pm.row_base + row] = d > 0.0f ? (M + log2f(d)) * kLn2 : -INFINITY;
  }
  named_bar_sync(kMergeBar, kMergeThreads);
}

// One pass of the in-kernel merge (kBlocks = 1 or 2): output dims dim_lo ..
// dim_lo + 64 * kBlocks - 1 of a unit from its n parts, as the segment merge does [vLLM #51705,
// 实现拆解 4, merge_mla_segments_triton]: out = sum_s 2^(m_s - M) acc_s / den.
// Thread t takes dim dim_lo + t % D (D = 64 kBlocks) for the row octets
// (t / D) * 8 / G .. (one 16-byte load per octet and part from the part's
// row-octet-major block; a warp's load covers D >= 64 consecutive dims of one
// octet, whole 128-byte runs).  Every part of a unit holds a token of its
// longest row, and rows without one in a part hold zeros there, so no
// liveness pass is needed: a zero weight selects 0.
template <int kBlocks>
__device__ void merge_unit_pass(const Params &p, const PendMerge &pm, int dim_lo, int tid, MergeScratch &ms) {
  constexpr int D = 64 * kBlocks;      // dims of this pass
  constexpr int G = kMergeThreads / D; // thread groups over the row octets
  constexpr int OP = 8 / G;            // octets per thread
  constexpr int BATCH = 16 / OP;       // parts whose loads are in flight at once
  const int S = p.num_segments, n = pm.n_parts;
  const int dl = tid % D, grp = tid / D;
  const int dim = dim_lo + dl;
  const float *mx = p.segm_max + static_cast<int64_t>(pm.row_base) * S;
  const int64_t blk0 = (static_cast<int64_t>(pm.b) * p.row_blocks + pm.rb) * S;
  float a[OP * 8];
#pragma unroll
  for (int k = 0; k < OP * 8; ++k) a[k] = 0.0f;
  for (int c0 = 0; c0 < n; c0 += kMergeSlots) {
    const int nc = min(kMergeSlots, n - c0);
    for (int i = tid; i < nc * kRows; i += kMergeThreads) {  // normalised weights of these parts
      const int sc = i / kRows, rr = i % kRows;
      float w = 0.0f;
      if (rr < pm.n_rows && ms.M[rr] != -INFINITY) {
        const float m = c0 == 0 ? ms.m[sc][rr] : __ldcg(mx + rr * S + c0 + sc);
        if (m != -INFINITY) w = exp2f(m - ms.M[rr]) * ms.inv[rr];
      }
      ms.w[sc][rr] = w;
    }
    named_bar_sync(kMergeBar, kMergeThreads);
    for (int i0 = 0; i0 < nc; i0 += BATCH) {
      uint4 x[BATCH][OP];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        if (i0 + u < nc) {
          const uint4 *blk = reinterpret_cast<const uint4 *>(p.segm_out + (blk0 + c0 + i0 + u) * (512 * kRows));
#pragma unroll
          for (int o = 0; o < OP; ++o) x[u][o] = __ldcg(blk + (grp * OP + o) * 512 + dim);
        }
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        if (i0 + u >= nc) break;
#pragma unroll
        for (int o = 0; o < OP; ++o) {
          const int r0 = 8 * (grp * OP + o);
          const float4 wa = *reinterpret_cast<const float4 *>(&ms.w[i0 + u][r0]);
          const float4 wb = *reinterpret_cast<const float4 *>(&ms.w[i0 + u][r0 + 4]);
          const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
          const uint32_t vv[4] = {x[u][o].x, x[u][o].y, x[u][o].z, x[u][o].w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // a weight of 0 selects 0
            const float e = __uint_as_float((k & 1) ? (vv[k >> 1] & 0xffff0000u) : (vv[k >> 1] << 16));
            a[8 * o + k] += (w[k] != 0.0f) ? w[k] * e : 0.0f;
          }
        }
      }
    }
    named_bar_sync(kMergeBar, kMergeThreads);  // weights are refilled by the next 32 parts
  }
  // [row][dim] through shared memory, then the rows' D dims out in 16-byte pieces
#pragma unroll
  for (int o = 0; o < OP; ++o)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __nv_bfloat16 hv = __float2bfloat16_rn(a[8 * o + k]);
      ms.o[8 * (grp * OP + o) + k][dl] = *reinterpret_cast<const uint16_t *>(&hv);
    }
  named_bar_sync(kMergeBar, kMergeThreads);
  constexpr int kPieces = kRows * D / 8;  // 16-byte pieces of the pass
  for (int i = tid; i < kPieces; i += kMergeThreads) {
    const int r = i / (D / 8), c16 = i % (D / 8);
    if (r < pm.n_rows) {
      const uint4 v = *reinterpret_cast<const uint4 *>(&ms.o[r][8 * c16]);
      *reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(pm.row_base) + r) * 512 + dim_lo + 8 * c16) = v;
    }
  }
  named_bar_sync(kMergeBar, kMergeThreads);  // scratch is reused by the next pass
}

// Merges a staged unit's claimed run of dims from shared memory (statistics
// already in ms, copies complete): passes of up to 128 dims, thread t taking
// dim t % Dp of the pass for the row octets (t / Dp) * 8 / G .., weights from
// ms.w (a zero weight selects 0), then the rows out in 16-byte pieces.
__device__ void merge_unit_from_stage(const Params &p, const PendMerge &pm, const uint8_t *stage, int tid,
                                      MergeScratch &ms) {
  int b0, nb;
  todo_run(pm.todo, b0, nb);
  const int D = 64 * nb, n = pm.n_parts;
  const uint4 *st = reinterpret_cast<const uint4 *>(stage + pm.staged);
  for (int pass0 = 0; pass0 < D; pass0 += 128) {
    const int Dp = min(128, D - pass0);  // 128 or 64
    const int G = kMergeThreads / Dp;    // 2 or 4 row-octet groups
    const int OP = 8 / G;                // 4 or 2 octets per thread
    const int dl = tid % Dp, grp = tid / Dp;
    float a[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) a[k] = 0.0f;
    for (int u = 0; u < n; ++u) {
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        if (o >= OP) break;
        const int oc = grp * OP + o;
        const uint4 xv = st[(u * 8 + oc) * D + pass0 + dl];
        const float4 wa = *reinterpret_cast<const float4 *>(&ms.w[u][8 * oc]);
        const float4 wb = *reinterpret_cast<const float4 *>(&ms.w[u][8 * oc + 4]);
        const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        const uint32_t vv[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // a weight of 0 selects 0
          const float e = __uint_as_float((k & 1) ? (vv[k >> 1] & 0xffff0000u) : (vv[k >> 1] << 16));
          a[8 * o + k] += (w[k] != 0.0f) ? w[k] * e : 0.0f;
        }
      }
    }
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      if (o >= OP) break;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __nv_bfloat16 hv = __float2bfloat16_rn(a[8 * o + k]);
        ms.o[8 * (grp * OP + o) + k][dl] = *reinterpret_cast<const uint16_t *>(&hv);
      }
    }
    named_bar_sync(kMergeBar, kMergeThreads);
    const int pieces = kRows * Dp / 8;
    for (int i = tid; i < pieces; i += kMergeThreads) {
      const int r = i / (Dp / 8), c16 = i % (Dp / 8);
      if (r < pm.n_rows) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&ms.o[r][8 * c16]);
        *reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(pm.row_base) + r) * 512 + 64 * b0 + pass0 + 8 * c16) = v;
      }
    }
    named_bar_sync(kMergeBar, kMergeThreads);  // ms.o is reused by the next pass
  }
}

// The normalised weights of a unit's first 32 parts into ms.w (statistics in ms).
__device__ void merge_unit_weights(const PendMerge &pm, int tid, MergeScratch &ms) {
  const int nc = min(kMergeSlots, pm.n_parts);
  for (int i = tid; i < nc * kRows; i += kMergeThreads) {
    const int sc = i / kRows, rr = i % kRows;
    float w = 0.0f;
    if (rr < pm.n_rows && ms.M[rr] != -INFINITY) {
      const float m = ms.m[sc][rr];
      if (m != -INFINITY) w = exp2f(m - ms.M[rr]) * ms.inv[rr];
    }
    ms.w[sc][rr] = w;
  }
  named_bar_sync(kMergeBar, kMergeThreads);
}

// Merges the 64-dim output blocks in pm.todo (bit k: dims 64k .. 64k+63) of
// one unit: the statistics once, then runs of consecutive blocks in passes
// of two blocks or one.  The LSE is written by whoever merges block 0.
__device__ void merge_unit(const Params &p, const PendMerge &pm, int tid, MergeScratch &ms) {
  merge_unit_stats(p, pm, (pm.todo & 1u) != 0, tid, ms);
  unsigned todo = pm.todo;
  while (todo != 0) {
    const int b0 = __ffs(todo) - 1;
    int run = 0;
    while (b0 + run < 8 && ((todo >> (b0 + run)) & 1u)) ++run;
    const int take = run >= 2 ? 2 : 1;
    if (take == 2) merge_unit_pass<2>(p, pm, 64 * b0, tid, ms);
    else merge_unit_pass<1>(p, pm, 64 * b0, tid, ms);
    todo &= ~(((1u << take) - 1u) << b0);
  }
}

template <bool kFp8, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the shared-window address (the 128-byte swizzle
  // pattern repeats every 1024 bytes and the descriptors assume that phase).
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc &misc = *reinterpret_cast<Misc *>(smem + kOffMisc);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_stage0 = s_base + kOffStages;   // stage s: + s * kStageBytes
  const uint32_t s_q = s_base + kOffQ;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.num_segments;
  const int P = p.page_size;
  const bool direct = (S == 1);
  constexpr bool fused = kFused;  // balanced split merged in this kernel (MLA_DECODE_FUSED_MERGE)

  // ---- setup: TMEM, barriers
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&misc.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&misc.full[i]), 1);
      mbar_init(smem_u32(&misc.ready[i]), kNumSoftmaxWarps);
      mbar_init(smem_u32(&misc.empty[i]), 1);
      mbar_init(smem_u32(&misc.s_full[i]), 1);
      mbar_init(smem_u32(&misc.p_full[i]), kNumSoftmaxWarps);
      mbar_init(smem_u32(&misc.o_done[i]), 1);
    }
    mbar_init(smem_u32(&misc.q_full), 1);
    mbar_init(smem_u32(&misc.q_empty), 1);
    mbar_init(smem_u32(&misc.fin), 1);
    for (int i = 0; i < kWorkRing; ++i) {
      mbar_init(smem_u32(&misc.work_full[i]), 1);
      mbar_init(smem_u32(&misc.work_empty[i]), 1 + kNumSoftmaxWarps);
    }
    misc.abort = 0;
    misc.n_pend = 0;
    fence_mbar_init();
  }
  // Nothing above touched global memory: the previous kernel in the stream
  // (which may produce this call's inputs, or read what it overwrites) has
  // completed from here on.
  grid_dep_wait();
  grid_dep_launch();
  const bool balanced = p.balanced != 0;
  // Balanced split: the producer's one chunk.  With the merge in this kernel
  // it is claimed from the work counter (a holder waits only for chunks that
  // running CTAs have claimed), the claim issued now so that its round trip
  // overlaps the unit table below; otherwise CTA c takes chunk c (every
  // chunk has a CTA: there are at most as many chunks as CTAs).
  int first_claim = static_cast<int>(blockIdx.x);
  if (kFused && balanced && warp == kProducerWarp && lane == 0) first_claim = atomicAdd(p.sched, 1);
  if (balanced) {
    // tiles of every (view, request, row block) unit: the request's longest
    // visible length in 64-token tiles, 0 for a row block without rows
    const int n_vb = p.num_views * p.num_reqs;
    for (int vb = threadIdx.x; vb < n_vb; vb += kThreads) {
      const int v = vb / p.num_reqs, b = vb % p.num_reqs;
      const int len = request_len(p, v, b);
      const int rows = len > 0 ? (p.qo_indptr[b + 1] - p.qo_indptr[b]) * p.num_heads : 0;
      const int t = (len + kTileTok - 1) / kTileTok;
      for (int rb = 0; rb < p.row_blocks; ++rb) misc.unit_end[vb * p.row_blocks + rb] = rb * kRows < rows ? t : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc.tmem_base;
  volatile int *abort_flag = &misc.abort;
  const long long budget = p.wait_budget;

  auto fail = [&](void) {
    *abort_flag = 1;
    record_error(p.err, MLA_DEV_WAIT_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // ======================================================== producer warp
    // Takes its chunk (balanced split) or claims work items (atomic
    // counter), publishes the entries to the other roles through the work
    // ring, and issues each entry's TMA loads: Q once, then every tile into
    // the next free stage.
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kv);
    }
    // A tile is loaded as runs of `run` consecutive cache rows (one sub-page,
    // or half of a 128-row sub-page), one box per run and chunk.
    const bool tile3d = p.tile3d != 0;
    const int run = P < kTileTok ? P : kTileTok;
    const int box_bytes = run * (kFp8 ? 64 : 128);
    // A stage is refilled only after its previous tile was consumed, so at
    // most one load per stage is in flight: remember the latest one (and the
    // latest Q load), for the exit path.
    uint32_t armed = 0, armed_par = 0;
    bool q_armed = false;
    uint32_t q_par = 0;
    uint32_t g = 0, kq = 0;  // running tile / Q-load counters
    bool ok = true;
    // Longest items first (the tail of the dynamic schedule is set by the
    // last long item claimed): with few enough requests every CTA ranks them
    // by their longest row (a request's rows are nondecreasing, so its last
    // row), ties by index, and claims in that order.
    const int *order = nullptr;
    if (!balanced && p.num_reqs <= kMaxOrderedReqs) {
      for (int b = lane; b < p.num_reqs; b += 32) {
        const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
        misc.req_key[b] = (q0 >= 0 && q1 > q0 && q1 <= p.num_rows) ? p.row_len[q1 - 1] : 0;
      }
      __syncwarp();
      for (int b = lane; b < p.num_reqs; b += 32) {
        const int key = misc.req_key[b];
        int rank = 0;
        for (int b2 = 0; b2 < p.num_reqs; ++b2) {
          const int k2 = misc.req_key[b2];
          rank += (k2 > key) || (k2 == key && b2 < b);
        }
        misc.req_order[rank] = b;
      }
      __syncwarp();
      order = misc.req_order;
    }
    // Balanced split: every unit with tiles is one overhead position (the
    // part's Q load and epilogue cost about one tile) followed by its tiles;
    // the V positions of all units laid end to end are cut into n chunks,
    // chunk c = [floor(c V / n), floor((c+1) V / n)), one per CTA (n smaller
    // when that keeps every unit within S chunks); a chunk's part of each
    // unit whose tiles it meets is one segment of that unit, numbered by
    // chunk from the unit's first.
    const int n_units = p.num_units;
    int T = 0, n_chunks = 0;  // T: V, the positions (tiles + overheads)
    if (balanced) {
      int carry = 0, tmax = 0;
      for (int base = 0; base < n_units; base += 32) {  // inclusive prefix sum, in place
        const int u = base + lane;
        const int t = u < n_units ? misc.unit_end[u] : 0;
        tmax = max(tmax, t);
        int x = t > 0 ? t + 1 : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (u < n_units) misc.unit_end[u] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      __syncwarp();
      T = carry;
      // chunks of at least `need` tiles meet at most S chunks per unit (S >= 2 here)
      const int need = max((tmax + S - 2) / (S - 1), 1);
      n_chunks = T > 0 ? min(static_cast<int>(gridDim.x), max(T / need, 1)) : 1;
    }
    // chunk holding position x (T > 0)
    auto chunk_of = [&](int x) {
      return static_cast<int>((static_cast<long long>(x + 1) * n_chunks - 1) / T);
    };
    // Each CTA claims one chunk at most (n_chunks <= grid): a chunk then
    // holds at most two multi-part units, its first and its last.
    int chunk = -1, c_lo = 0, c_hi = 0, c_hi_ext = 0, u_next = 0;
    bool claimed = false;
    for (uint32_t k = 0;; ++k) {
      const uint32_t ws = k % kWorkRing;
      WorkEntry &e = misc.work[ws];
      if (lane == 0 && ok &&
          !mbar_wait(smem_u32(&misc.work_empty[ws]), ((k / kWorkRing) & 1u) ^ 1u, abort_flag, budget)) {
        fail();
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      // the next part: (view, request, row block), segment slot, tile range
      bool done = !ok;
      int w = 0, v = 0, b = 0, rb = 0, seg = 0, fill_hi = 0, t_a = 0, t_b = 0, u_start = 0;
      int unit = 0, n_parts = 0, c_last = 0;
      if (!done && balanced) {
        while (true) {
          if (chunk < 0) {
            if (claimed) {
              done = true;
              break;
            }
            claimed = true;
            const int c = __shfl_sync(0xffffffffu, first_claim, 0);
            if (c >= n_chunks) {
              done = true;
              break;
            }
            chunk = c;
            c_lo = static_cast<int>(static_cast<long long>(c) * T / n_chunks);
            c_hi = static_cast<int>(static_cast<long long>(c + 1) * T / n_chunks);
            c_hi_ext = c == n_chunks - 1 ? T + 1 : c_hi;  // units without tiles at the very end
            int u = 0, u_hi = n_units;  // first unit whose prefix reaches c_lo
            while (u < u_hi) {
              const int mid = (u + u_hi) >> 1;
              if (misc.unit_end[mid] < c_lo) u = mid + 1;
              else u_hi = mid;
            }
            u_next = u;
          }
          bool found = false;
          while (u_next < n_units) {
            const int u = u_next;
            const int end = misc.unit_end[u];
            const int prev = u == 0 ? 0 : misc.unit_end[u - 1];
            const int start = prev + (end > prev ? 1 : 0);  // first tile, past the overhead position
            if (start >= c_hi_ext) break;
            ++u_next;
            if (end > start && end <= c_lo) continue;  // all of its tiles lie before this chunk
            if (end == start) {  // no tiles: one empty part marks all its slots
              t_a = t_b = start;
              seg = 0;
              fill_hi = S;
              n_parts = 0;
              c_last = chunk;
            } else {
              t_a = max(c_lo, start);
              t_b = min(c_hi, end);
              seg = chunk - chunk_of(start);
              fill_hi = end <= c_hi ? S : seg + 1;  // its last part marks the slots no chunk reached
              c_last = chunk_of(end - 1);
              n_parts = c_last - chunk_of(start) + 1;
            }
            unit = u;
            u_start = start;
            const int vb = u / p.row_blocks;
            rb = u - vb * p.row_blocks;
            v = vb / p.num_reqs;
            b = vb - v * p.num_reqs;
            found = true;
            break;
          }
          if (found) break;
          chunk = -1;  // chunk exhausted: claim the next
        }
        w = chunk;
      } else if (!done) {
        if (lane == 0) w = atomicAdd(p.sched, 1);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (w >= p.num_items) {
          done = true;
        } else {
          // item order: request (longest first), then view, row block, segment
          seg = w % S;
          fill_hi = seg + 1;
          rb = (w / S) % p.row_blocks;
          v = (w / (S * p.row_blocks)) % p.num_views;
          const int ob = w / (S * p.row_blocks * p.num_views);
          b = order != nullptr ? order[ob] : ob;
        }
      }
      if (done) {
        if (lane == 0) {
          e.w = -1;
          mbar_arrive(smem_u32(&misc.work_full[ws]));
        }
        break;
      }
      bool clipped = false;
      int group_len = 0;
      const bool good = decode_unit(p, v, b, rb, e, lane, clipped, group_len);
      __syncwarp();
      if (lane == 0) {
        e.w = w;
        e.seg = seg;
        e.fill_hi = fill_hi;
        e.unit = unit;
        e.n_parts = n_parts;
        e.c_last = c_last;
        if (balanced) {
          e.seg_lo = (t_a - u_start) * kTileTok;
          e.seg_hi = min((t_b - u_start) * kTileTok, group_len);
        } else {
          const long long span = static_cast<long long>(S) * P;
          const int seg_tokens = static_cast<int>((group_len + span - 1) / span) * P;
          e.seg_lo = seg * seg_tokens;
          e.seg_hi = min(e.seg_lo + seg_tokens, group_len);
        }
        e.n_tiles = (e.n_rows > 0 && e.seg_lo < e.seg_hi) ? (e.seg_hi - e.seg_lo + kTileTok - 1) / kTileTok : 0;
        if (!good) {
          record_error(p.err, MLA_DEV_BAD_INDPTR);
          e.n_rows = 0;
          e.n_tiles = 0;
        }
        if (clipped) record_error(p.err, MLA_DEV_LEN_BOUND);
        mbar_arrive(smem_u32(&misc.work_full[ws]));
      }
      const int n_tiles = __shfl_sync(0xffffffffu, lane == 0 ? e.n_tiles : 0, 0);
      if (n_tiles > 0) {
        const int seg_lo = e.seg_lo, seg_hi = e.seg_hi, q_row = e.q_row;
        // Sub-page ids are read 32 at a time (lane l holds page win_base + l),
        // ahead of the waits, so no id fetch sits between a freed stage and
        // its next copies.
        const int32_t *sp_row = p.subpage_table + static_cast<int64_t>(e.b) * p.subpage_stride;
        const int last_page = (seg_hi - 1) / P;
        int win_base = seg_lo / P;
        int32_t win_id = (win_base + lane <= last_page) ? sp_row[win_base + lane] : -1;
        // Q of this item, once the previous item's last QK is done with the buffer
        if (lane == 0 && ok &&
            !mbar_wait(smem_u32(&misc.q_empty), (kq & 1u) ^ 1u, abort_flag, budget)) {
          fail();
          ok = false;
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        const uint32_t q_bar = smem_u32(&misc.q_full);
        if (ok) {
          if (lane == 0) mbar_arrive_expect_tx(q_bar, kNumChunks * kQChunkBytes);
          __syncwarp();
          if (lane < kNumChunks)
            tma_load_2d(s_q + lane * kQChunkBytes, &tm_q, q_bar, lane * 64, q_row, pol_q);
          q_armed = true;
          q_par = kq & 1u;
        }
        ++kq;
        for (int i = 0; i < n_tiles && ok; ++i, ++g) {
          const int tok0 = seg_lo + i * kTileTok;
          const int n_valid = min(kTileTok, seg_hi - tok0);
          const int n_ops = ((n_valid + run - 1) / run) * kNumChunks;
          const uint32_t st = g & 1u;
          if ((tok0 + n_valid - 1) / P >= win_base + 32) {  // warp-uniform: slide the id window
            win_base = tok0 / P;
            win_id = (win_base + lane <= last_page) ? sp_row[win_base + lane] : -1;
          }
          if (lane == 0 && !mbar_wait(smem_u32(&misc.empty[st]), ((g >> 1) & 1u) ^ 1u, abort_flag, budget)) {
            fail();
            ok = false;
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          const uint32_t fbar = smem_u32(&misc.full[st]);
          // fp8 codes land packed in the stage's upper half (chunk c at c * 4 KB)
          const uint32_t dst0 = s_stage0 + st * kStageBytes + (kFp8 ? kStageBytes / 2 : 0);
          if (tile3d) {
            // P >= 64: the tile is 64 consecutive rows of one sub-page, one 3-D box
            const int32_t id = __shfl_sync(0xffffffffu, win_id, tok0 / P - win_base);
            if (lane == 0) {
              int32_t row;
              if (id < 0 || static_cast<int64_t>(id) * P + P > p.num_cache_rows) {
                record_error(p.err, MLA_DEV_BAD_SUBPAGE);
                row = static_cast<int32_t>(p.num_cache_rows);  // out of range: zero fill
              } else {
                row = id * P + (tok0 % P);
              }
              mbar_arrive_expect_tx(fbar, kFp8 ? kStageBytes / 2 : kStageBytes);
              tma_load_3d(dst0, &tm_kv, fbar, 0, row, 0, pol_kv);
            }
            armed |= 1u << st;
            armed_par = (armed_par & ~(1u << st)) | (((g >> 1) & 1u) << st);
            continue;
          }
          if (lane == 0) mbar_arrive_expect_tx(fbar, n_ops * box_bytes);
          __syncwarp();  // the expected bytes are posted before any copy can complete
          for (int o0 = 0; o0 < n_ops; o0 += 32) {  // uniform trip count (the shuffle needs every lane)
            const int o = o0 + lane;
            const int r = o / kNumChunks, c = o - r * kNumChunks;
            const int t = tok0 + r * run;
            const int src = o < n_ops ? t / P - win_base : 0;
            const int32_t id = __shfl_sync(0xffffffffu, win_id, src);
            if (o < n_ops) {
              int32_t row;
              if (id < 0 || static_cast<int64_t>(id) * P + P > p.num_cache_rows) {
                record_error(p.err, MLA_DEV_BAD_SUBPAGE);
                row = static_cast<int32_t>(p.num_cache_rows);  // out of range: zero fill
              } else {
                row = id * P + (t % P);
              }
              tma_load_2d(dst0 + c * (kFp8 ? kChunkBytes / 2 : kChunkBytes) + r * box_bytes, &tm_kv, fbar,
                          c * 64, row, pol_kv);
            }
          }
          armed |= 1u << st;
          armed_par = (armed_par & ~(1u << st)) | (((g >> 1) & 1u) << st);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    if (lane == 0 && (!ok || *abort_flag)) {
      // Let the copies already issued land before the CTA's memory is
      // released (a copy completes by itself; this wait has its own budget).
      const volatile int never = 0;
      for (int st = 0; st < kStages; ++st)
        if (armed & (1u << st))
          mbar_wait(smem_u32(&misc.full[st]), (armed_par >> st) & 1u, &never, p.drain_budget);
      if (q_armed) mbar_wait(smem_u32(&misc.q_full), q_par, &never, p.drain_budget);
    }
  } else if (warp == kMmaWarp) {
    // ======================================================== UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kTileTok, kRows, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kRows, 1, 1);
      // Descriptors are built once; the start-address field (address >> 4 in
      // the low 14 bits, addresses < 256 KB) is advanced with integer adds.
      //   K chunk c of stage s:  d_k0 + s * 4608 + c * 512   (+2 per 16 dims)
      //   Q chunk c:             d_q0 + c * 512
      //   V^T block b:           d_v0 + s * 4608 + b * 1024  (LBO: next 64-dim chunk; +128 per 16 tokens)
      //   P^T (rope chunk):      d_p0 + s * 4608             (+128 per 16 tokens)
      constexpr uint32_t kStageDesc = kStageBytes >> 4;
      const uint64_t d_k0 = sdesc_sw128(s_stage0, 0, 1024);
      const uint64_t d_q0 = sdesc_sw128(s_q, 0, 1024);
      const uint64_t d_v0 = sdesc_sw128(s_stage0, kChunkBytes, 1024);
      const uint64_t d_p0 = sdesc_sw128(s_stage0 + kPChunk * kChunkBytes, kChunkBytes, 1024);
      // Event loop: PV of the oldest tile whose P^T is ready goes first (it
      // frees that tile's stage for the next load); otherwise the next work
      // entry, the item's Q, or QK of the item's next tile once its data has
      // landed and an S^T buffer is free (at most two tiles between QK and
      // PV).  Polling uses non-blocking barrier tests.
      uint32_t gq = 0, gp = 0, kq = 0, k = 0;  // tiles QK'd / PV'd, Q loads, work entries
      uint32_t first_bits = 0, last_bits = 0, k16_bits = 0;  // per S^T buffer: first / last tile of its item, 16-token steps
      int it_left = 0, it_i = 0, it_lo = 0, it_hi = 0;
      uint32_t grace_g = 0xffffffffu;  // tile whose QK already waited for a pending PV
      bool q_ready = false, no_more = false;
      long long idle_since = clock64();
      while (true) {
        bool progress = true;
        if (gp < gq && mbar_test(smem_u32(&misc.p_full[gp & 1u]), (gp >> 1) & 1u)) {
          tc_fence_after();
          const uint32_t st = gp & 1u;
          const bool first = (first_bits >> st) & 1u;
          const int n_k16 = static_cast<int>((k16_bits >> (4 * st)) & 15u);
          const uint64_t dv = d_v0 + st * kStageDesc, dp = d_p0 + st * kStageDesc;
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t t_o = tmem + kTmemO + blk * kRows;
            const uint64_t da = dv + static_cast<uint64_t>(blk) * ((2 * kChunkBytes) >> 4);
            if (first) umma_bf16_ss_first(t_o, da, dp, idesc_pv);
            else umma_bf16_ss_acc(t_o, da, dp, idesc_pv);
#pragma unroll
            for (int kk = 1; kk < kTileTok / 16; ++kk)
              if (kk < n_k16) umma_bf16_ss_acc(t_o, da + kk * 128, dp + kk * 128, idesc_pv);
          }
          umma_commit(smem_u32(&misc.o_done[st]));
          umma_commit(smem_u32(&misc.empty[st]));  // stage (V and P^T) free for the next load
          ++gp;
        } else if (it_left == 0 && !no_more) {
          const uint32_t ws = k % kWorkRing;
          if (mbar_test(smem_u32(&misc.work_full[ws]), (k / kWorkRing) & 1u)) {
            const WorkEntry &e = misc.work[ws];
            const int w = e.w;
            it_left = w >= 0 ? e.n_tiles : 0;
            it_lo = e.seg_lo;
            it_hi = e.seg_hi;
            it_i = 0;
            q_ready = false;
            if (w >= 0) mbar_arrive(smem_u32(&misc.work_empty[ws]));
            else no_more = true;
            ++k;
          } else {
            progress = false;
          }
        } else if (it_left > 0 && !q_ready) {
          if (mbar_test(smem_u32(&misc.q_full), kq & 1u)) {
            ++kq;
            q_ready = true;
            tc_fence_after();
          } else {
            progress = false;
          }
        } else if (it_left > 0 && gq - gp < 2 &&
                   mbar_test(smem_u32(kFp8 ? &misc.ready[gq & 1u] : &misc.full[gq & 1u]), (gq >> 1) & 1u)) {
          // The tensor pipe runs UMMAs in issue order, and QK of a tile keeps
          // it busy for about a microsecond.  A PV whose P^T is about to be
          // ready (the softmax of that tile is under way) goes first: it
          // frees a stage for the next load.  Bounded grace period.
          if (gp < gq && grace_g != gq) {
            grace_g = gq;
            const long long grace = ((last_bits >> (gp & 1u)) & 1u) ? kPvGraceLast : kPvGrace;
            const long long t0 = clock64();
            while (!mbar_test(smem_u32(&misc.p_full[gp & 1u]), (gp >> 1) & 1u) && clock64() - t0 < grace) {
            }
            continue;  // back to the top: the PV branch takes it if it is ready
          }
          tc_fence_after();
          const uint32_t st = gq & 1u;
          const uint32_t t_s = tmem + kTmemS + st * 64;
          const uint64_t dk = d_k0 + st * kStageDesc;
#pragma unroll
          for (int c = 0; c < kNumChunks; ++c) {
            const uint64_t da = dk + static_cast<uint64_t>(c) * (kChunkBytes >> 4);
            const uint64_t db = d_q0 + static_cast<uint64_t>(c) * (kQChunkBytes >> 4);
            if (c == 0) umma_bf16_ss_first(t_s, da, db, idesc_qk);
            else umma_bf16_ss_acc(t_s, da, db, idesc_qk);
            umma_bf16_ss_acc(t_s, da + 2, db + 2, idesc_qk);  // +32 bytes along K
            umma_bf16_ss_acc(t_s, da + 4, db + 4, idesc_qk);
            umma_bf16_ss_acc(t_s, da + 6, db + 6, idesc_qk);
          }
          if (it_left == 1) umma_commit(smem_u32(&misc.q_empty));  // Q free for the next item
          umma_commit(smem_u32(&misc.s_full[st]));
          const int n_valid = min(kTileTok, it_hi - (it_lo + it_i * kTileTok));
          first_bits = (first_bits & ~(1u << st)) | (static_cast<uint32_t>(it_i == 0) << st);
          last_bits = (last_bits & ~(1u << st)) | (static_cast<uint32_t>(it_left == 1) << st);
          k16_bits = (k16_bits & ~(15u << (4 * st))) | (static_cast<uint32_t>((n_valid + 15) / 16) << (4 * st));
          ++gq;
          ++it_i;
          --it_left;
        } else {
          progress = false;
        }
        if (no_more && it_left == 0 && gp == gq) break;
        if (progress) {
          idle_since = clock64();
        } else if (*abort_flag || clock64() - idle_since > budget) {
          fail();
          break;
        }
      }
      umma_commit(smem_u32(&misc.fin));  // every MMA issued so far has retired
      const volatile int never = 0;
      mbar_wait(smem_u32(&misc.fin), 0, &never, p.drain_budget);
    }
  } else {
    // ======================================================== softmax warps
    const int g_col = warp >> 2;       // column group: rows 32g .. 32g+31 of the block
    const int wq = warp & 3;           // TMEM lane quarter
    // S^T (M = 64) puts token 16 q + i in TMEM lane 32 q + i: this thread
    // handles token `tok` and the 16 columns 32g + 16h .. 32g + 16h + 15.
    const int half = lane >> 4;
    const int tok = wq * 16 + (lane & 15);
    const int dim_lane = wq * 32 + lane;    // dim row of an O^T block
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const int my_col = 32 * g_col + lane;  // column whose statistics this lane keeps
    int red_buf = 0;
    bool ok = true;
    uint32_t g = 0;

    for (uint32_t k = 0;; ++k) {
      const uint32_t ws = k % kWorkRing;
      if (ok && !mbar_wait(smem_u32(&misc.work_full[ws]), (k / kWorkRing) & 1u, abort_flag, budget)) {
        fail();
        ok = false;
      }
      // All softmax warps take the same exit decision (they share named
      // barriers below): one thread snapshots it between two barriers.
      named_bar_sync(4, kNumSoftmaxWarps * 32);
      if (threadIdx.x == 0) misc.sm_stop[k & 1u] = (*abort_flag != 0) || (misc.work[ws].w < 0);
      named_bar_sync(4, kNumSoftmaxWarps * 32);
      if (misc.sm_stop[k & 1u]) break;
      const WorkEntry &e = misc.work[ws];
      const int n_rows = e.n_rows, n_tiles = e.n_tiles, seg = e.seg, e_b = e.b, e_rb = e.rb, fill_hi = e.fill_hi;
      const int row_base = e.row_base, seg_lo = e.seg_lo, seg_hi = e.seg_hi;
      const int n_parts = e.n_parts, c_last = e.c_last, e_unit = e.unit;
      // normalised bf16 rows + LSE straight from TMEM: one segment, or (in-kernel
      // merge) a unit whose tiles all lie in this CTA's chunk
      const bool to_out = direct || (fused && n_parts == 1);
      if (n_rows > 0 && n_tiles == 0) {
        // nothing visible in this segment for any row of the block
        if (wq == 0 && my_col < n_rows) {
          const int64_t r = row_base + my_col;
          if (direct || fused) {
            p.lse[r] = -INFINITY;
          } else {
            for (int s2 = seg; s2 < max(fill_hi, seg + 1); ++s2) {
              p.segm_max[r * S + s2] = -INFINITY;
              p.segm_sum[r * S + s2] = 0.0f;
            }
          }
        }
        if ((direct || fused) && my_col < n_rows) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.out + (row_base + my_col) * 512);
          for (int ee = wq; ee < 64; ee += 4) dst[ee] = make_uint4(0, 0, 0, 0);
        }
      }
      if (n_tiles == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&misc.work_empty[ws]));
        continue;
      }
      // this thread's 16 columns' visible lengths, constant over the entry's tiles
      int lv[16];
      {
        const int *lens_h = &e.lens[32 * g_col + 16 * half];
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const int4 l4 = *reinterpret_cast<const int4 *>(&lens_h[4 * j4]);
          lv[4 * j4 + 0] = l4.x;
          lv[4 * j4 + 1] = l4.y;
          lv[4 * j4 + 2] = l4.z;
          lv[4 * j4 + 3] = l4.w;
        }
      }
      float l_part[16];
      float m_col[16];  // reference max of this thread's 16 columns (lane c keeps m_ref of group column c)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        l_part[j] = 0.0f;
        m_col[j] = -INFINITY;
      }
      float m_ref = -INFINITY;

      for (int i = 0; i < n_tiles; ++i, ++g) {
        const int tok0 = seg_lo + i * kTileTok;
        const int n_valid = min(kTileTok, seg_hi - tok0);
        const uint32_t st = g & 1u;
        const uint32_t par = (g >> 1) & 1u;
        const uint32_t s_stage = s_stage0 + st * kStageBytes;

        if constexpr (kFp8) {
          // Expand the stage's nine fp8 chunks (packed in its upper half) to
          // bf16 in place: every thread reads its 16 codes of each chunk,
          // then all write.
          if (ok && !mbar_wait(smem_u32(&misc.full[st]), par, abort_flag, budget)) {
            fail();
            ok = false;
          }
          const int t4 = threadIdx.x >> 2;  // token row 0..63
          const int qt = threadIdx.x & 3;   // which 16 of the 64 dims
          uint4 raw[kNumChunks];
#pragma unroll
          for (int c = 0; c < kNumChunks; ++c)
            raw[c] = ld_shared_v4(s_stage + kStageBytes / 2 + c * (kChunkBytes / 2) + t4 * 64 + qt * 16);
          named_bar_sync(3, kNumSoftmaxWarps * 32);
#pragma unroll
          for (int c = 0; c < kNumChunks; ++c) {
            const uint32_t row_addr = s_stage + c * kChunkBytes + t4 * 128;
            const uint32_t c0 = static_cast<uint32_t>((2 * qt) ^ (t4 & 7));
            const uint32_t c1 = static_cast<uint32_t>((2 * qt + 1) ^ (t4 & 7));
            st_shared_v4(row_addr + c0 * 16, e4m3x2_to_bf16x2(raw[c].x & 0xffff), e4m3x2_to_bf16x2(raw[c].x >> 16),
                         e4m3x2_to_bf16x2(raw[c].y & 0xffff), e4m3x2_to_bf16x2(raw[c].y >> 16));
            st_shared_v4(row_addr + c1 * 16, e4m3x2_to_bf16x2(raw[c].z & 0xffff), e4m3x2_to_bf16x2(raw[c].z >> 16),
                         e4m3x2_to_bf16x2(raw[c].w & 0xffff), e4m3x2_to_bf16x2(raw[c].w >> 16));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&misc.ready[st]));
        }

        if (ok && !mbar_wait(smem_u32(&misc.s_full[st]), par, abort_flag, budget)) {
          fail();
          ok = false;
        }
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16x2(tmem + lane_addr + kTmemS + st * 64 + 32 * g_col, sv);

        // scaled scores (log2 units), causal + segment mask per column
        float x[16];
        const int gtok = tok0 + tok;
        const bool tok_in = tok < n_valid;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          x[j] = (tok_in && gtok < lv[j]) ? __uint_as_float(sv[j]) * p.score_scale_log2 : -INFINITY;
        // The column max is needed only when some score exceeds the column's
        // reference by more than the lazy-rescale threshold (always on the
        // first tile that sees data).  One barrier-reduction votes per group.
        bool exceed = false;
#pragma unroll
        for (int j = 0; j < 16; ++j) exceed |= (x[j] - m_col[j] > kRescaleThreshold);
        const bool group_exceed = named_bar_red_or(1 + g_col, 128, exceed);
        bool any_rescale = false;
        float alpha = 1.0f;
        if (group_exceed) {
          float red[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) red[j] = x[j];
          const float wmax = half_reduce_scatter<true>(red, lane);  // column `lane` of the group
          misc.red[red_buf][g_col][wq][lane] = wmax;
          named_bar_sync(1 + g_col, 128);
          const float tmax =
              fmaxf(fmaxf(misc.red[red_buf][g_col][0][lane], misc.red[red_buf][g_col][1][lane]),
                    fmaxf(misc.red[red_buf][g_col][2][lane], misc.red[red_buf][g_col][3][lane]));
          red_buf ^= 1;
          if (tmax > m_ref + kRescaleThreshold) {
            alpha = fast_exp2(m_ref - tmax);  // 0 when m_ref is -inf
            m_ref = tmax;
          }
          any_rescale = __any_sync(0xffffffffu, alpha != 1.0f);
#pragma unroll
          for (int j = 0; j < 16; ++j) m_col[j] = __shfl_sync(0xffffffffu, m_ref, 16 * half + j);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)  // probability (0 for masked entries and empty columns)
          x[j] = (x[j] == -INFINITY) ? 0.0f : fast_exp2(x[j] - m_col[j]);
        if (any_rescale) {
#pragma unroll
          for (int j = 0; j < 16; ++j) l_part[j] *= __shfl_sync(0xffffffffu, alpha, 16 * half + j);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) l_part[j] += x[j];

        // P^T row `tok`, columns 32g + 16h .. +15 (bf16, 128-byte swizzle),
        // into the stage's rope chunk (the tile's QK has retired it).
        const uint32_t s_pt = s_stage + kPChunk * kChunkBytes;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t chunk = static_cast<uint32_t>((4 * g_col + 2 * half + q) ^ (tok & 7));
          st_shared_v4(s_pt + tok * 128 + chunk * 16, pack_bf16(x[8 * q + 0], x[8 * q + 1]),
                       pack_bf16(x[8 * q + 2], x[8 * q + 3]), pack_bf16(x[8 * q + 4], x[8 * q + 5]),
                       pack_bf16(x[8 * q + 6], x[8 * q + 7]));
        }
        // V rows past the last valid token but inside the last 16-token MMA
        // step hold stale or foreign data: zero them so 0 * V stays 0 (this
        // thread: two of the row's eight V chunks).
        if (tok >= n_valid && tok < ((n_valid + 15) & ~15)) {
          for (int c = 4 * g_col + 2 * half; c < 4 * g_col + 2 * half + 2; ++c)
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16)
              st_shared_v4(s_stage + c * kChunkBytes + tok * 128 + c16 * 16, 0, 0, 0, 0);
        }
        // O is rescaled only after the previous tile's PV retired.  o_done
        // has one barrier per stage, so a stage's completions are two tiles
        // apart: the wait for tile g-1 can neither see a stale phase nor one
        // two ahead (PV of tile g+1 needs this tile's P^T first).
        if (i > 0 && any_rescale) {
          if (ok && !mbar_wait(smem_u32(&misc.o_done[(g - 1) & 1u]), ((g - 1) >> 1) & 1u, abort_flag, budget)) {
            fail();
            ok = false;
          }
          tc_fence_after();
        }
        if (i > 0 && any_rescale) {
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t taddr = tmem + lane_addr + kTmemO + blk * kRows + 32 * g_col;
            uint32_t ov[32];
            tmem_ld32(taddr, ov);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              ov[j] = __float_as_uint(__uint_as_float(ov[j]) * __shfl_sync(0xffffffffu, alpha, j));
            tmem_st32(taddr, ov);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&misc.p_full[st]));
      }

      // ---- epilogue of the item: row sums and statistics (while the last
      // PV runs), then the output
      const float wsum = half_reduce_scatter<false>(l_part, lane);  // column `lane` of the group
      misc.red[red_buf][g_col][wq][lane] = wsum;
      named_bar_sync(1 + g_col, 128);
      const float l_tot = misc.red[red_buf][g_col][0][lane] + misc.red[red_buf][g_col][1][lane] +
                          misc.red[red_buf][g_col][2][lane] + misc.red[red_buf][g_col][3][lane];
      red_buf ^= 1;
      if (ok && wq == 0 && my_col < n_rows) {
        const int64_t r = row_base + my_col;
        if (to_out) {
          p.lse[r] = (l_tot > 0.0f) ? (m_ref + __log2f(l_tot)) * kLn2 : -INFINITY;
        } else {
          p.segm_max[r * S + seg] = (l_tot > 0.0f) ? m_ref : -INFINITY;
          p.segm_sum[r * S + seg] = l_tot;
          for (int s2 = seg + 1; s2 < fill_hi; ++s2) {  // slots of this unit that no part reaches
            p.segm_max[r * S + s2] = -INFINITY;
            p.segm_sum[r * S + s2] = 0.0f;
          }
        }
      }
      const float col_scale = (l_tot > 0.0f) ? (to_out ? p.out_scale / l_tot : p.out_scale) : 0.0f;
      const int n_cols = min(32, n_rows - 32 * g_col);
      // column j's scale (0: the row saw no token here) gathered once for all four blocks
      float sc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[j] = __shfl_sync(0xffffffffu, col_scale, j);
      const int64_t r0 = row_base + 32 * g_col;
      if (ok && !mbar_wait(smem_u32(&misc.o_done[(g - 1) & 1u]), ((g - 1) >> 1) & 1u, abort_flag, budget)) {
        fail();
        ok = false;
      }
      tc_fence_after();
      // O^T blocks two at a time: both TMEM loads in flight, one wait
#pragma unroll 1
      for (int b2 = 0; b2 < 4; b2 += 2) {
        uint32_t ovp[2][32];
        tmem_ld32_async(tmem + lane_addr + kTmemO + b2 * kRows + 32 * g_col, ovp[0]);
        tmem_ld32_async(tmem + lane_addr + kTmemO + (b2 + 1) * kRows + 32 * g_col, ovp[1]);
        tmem_wait_ld();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int blk = b2 + h2;
          const uint32_t (&ov)[32] = ovp[h2];
          if (!ok || *abort_flag != 0) continue;
          const int dim = blk * 128 + dim_lane;
          if (to_out) {
            __nv_bfloat16 *o = p.out + r0 * 512 + dim;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < n_cols) o[static_cast<int64_t>(j) * 512] = __float2bfloat16_rn(__uint_as_float(ov[j]) * sc[j]);
          } else {
            // partial block (b, rb, seg), [8 row octets][512 dims][8 rows]:
            // this thread's dim in the group's four octets, one 16-byte store
            // each; a warp's store covers 32 consecutive dims, 512 contiguous
            // bytes (a row that saw no token here gets 0)
            uint4 *o = reinterpret_cast<uint4 *>(
                           p.segm_out + ((static_cast<int64_t>(e_b) * p.row_blocks + e_rb) * S + seg) * (512 * kRows)) +
                       (4 * g_col) * 512 + dim;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w4[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int j = 8 * q + 2 * u;
                const float lo = sc[j] != 0.0f ? __uint_as_float(ov[j]) * sc[j] : 0.0f;
                const float hi = sc[j + 1] != 0.0f ? __uint_as_float(ov[j + 1]) * sc[j + 1] : 0.0f;
                w4[u] = pack_bf16(lo, hi);
              }
              o[q * 512] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
      tc_fence_before();  // O reads done before the next item's first PV overwrites O
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&misc.work_empty[ws]));
      if (fused && n_parts > 1 && threadIdx.x == 0) {
        // a part of a multi-part unit: published (and the unit merged) once
        // this CTA's own work is done
        if (misc.n_pend < kMaxPend) {
          PendMerge &pm = misc.pend[misc.n_pend++];
          pm.b = e_b;
          pm.rb = e_rb;
          pm.row_base = row_base;
          pm.n_rows = n_rows;
          pm.n_parts = n_parts;
          pm.unit = e_unit;
          pm.seg = seg;
          pm.c_last = c_last;
        } else {
          record_error(p.err, MLA_DEV_WAIT_TIMEOUT);  // cannot happen: one chunk per CTA
        }
      }
    }
    if (fused) {
      // The CTA's own parts are done: every tile's PV has retired and no copy
      // is in flight, so stage 0 is free for the merge scratch.  Publish the
      // parts: every thread's stores are fenced before the barrier, then one
      // release add per part counts it.  A holder that will wait for its
      // unit -- only when every chunk of the unit is claimed, i.e. held by a
      // running CTA, which publishes without waiting on anyone -- claims its
      // share of the eight 64-dim output blocks in the same add; the holder
      // of the last part to arrive merges every block nobody claimed.
      __threadfence();
      named_bar_sync(kMergeBar, kMergeThreads);
      const int n_pend = misc.n_pend;
      if (threadIdx.x == 0) {
        for (int i = 0; i < n_pend; ++i) {
          PendMerge &pm = misc.pend[i];
          // holder k of n takes the consecutive blocks [8k / n, 8(k+1) / n)
          const int blo = (8 * pm.seg) / pm.n_parts, bhi = (8 * (pm.seg + 1)) / pm.n_parts;
          const unsigned mine = ((1u << bhi) - 1u) & ~((1u << blo) - 1u);
          const bool can_wait = ld_volatile(p.sched) > pm.c_last;
          const unsigned add = 1u + (can_wait ? (mine << 16) : 0u);
          const unsigned old = atom_add_release_gpu(p.unit_state + pm.unit, add);
          const bool last = (old & 0xffffu) == static_cast<unsigned>(pm.n_parts - 1);
          pm.todo = last ? (~(old >> 16) & 0xffu) : (can_wait ? mine : 0u);
          pm.wait = last ? 0 : 1;
        }
      }
      // staging plan: a unit whose claim is one run of blocks and whose parts'
      // slices fit the remaining staging area is copied into shared memory
      // (all copies in flight at once); others are read from L2 directly
      if (threadIdx.x == 0) {
        int used = 0;
        for (int i = 0; i < n_pend; ++i) {
          PendMerge &pm = misc.pend[i];
          pm.staged = -1;
          if (pm.todo == 0 || pm.n_parts > kMergeSlots) continue;
          int b0, nb;
          todo_run(pm.todo, b0, nb);
          const int bytes = pm.n_parts * 8 * 64 * nb * 16;
          if (nb > 0 && used + bytes <= kStagingBytes) {
            pm.staged = used;
            used += bytes;
          }
        }
      }
      named_bar_sync(kMergeBar, kMergeThreads);
      fence_proxy_async_smem();
      MergeScratch &ms = *reinterpret_cast<MergeScratch *>(smem + kOffQ);
      const uint8_t *stage_gen = smem + kOffStages;
      // Two-step pipeline over the pending units: wait (bounded) for unit i
      // and issue its copies, then merge unit i - 1 while they fly.
      auto merge_pending = [&](int i, int later) {
        const PendMerge pm = misc.pend[i];
        if (pm.todo == 0 || !pm.go) return;
        __threadfence();
        if (pm.staged < 0) {
          merge_unit(p, pm, threadIdx.x, ms);
          return;
        }
        merge_unit_stats(p, pm, (pm.todo & 1u) != 0, threadIdx.x, ms);
        merge_unit_weights(pm, threadIdx.x, ms);
        if (later > 0) cp_async_wait<1>();
        else cp_async_wait<0>();
        named_bar_sync(kMergeBar, kMergeThreads);
        merge_unit_from_stage(p, pm, stage_gen, threadIdx.x, ms);
      };
      for (int i = 0; i < n_pend; ++i) {
        if (threadIdx.x == 0) {
          PendMerge &pm = misc.pend[i];
          bool go = pm.todo != 0 && ok && *abort_flag == 0;
          if (go && pm.wait) {  // bounded wait for the unit's other parts
            const long long t0 = clock64();
            while ((ld_acquire_gpu(p.unit_state + pm.unit) & 0xffffu) != static_cast<unsigned>(pm.n_parts)) {
              if (*abort_flag || clock64() - t0 > budget) {
                fail();
                go = false;
                break;
              }
              __nanosleep(64);
            }
          }
          pm.go = go ? 1 : 0;
        }
        __syncwarp();
        named_bar_sync(kMergeBar, kMergeThreads);
        if (misc.pend[i].go && misc.pend[i].staged >= 0) {
          __threadfence();
          stage_unit(p, misc.pend[i], s_stage0, threadIdx.x);
        }
        cp_async_commit();  // one group per pending unit (empty when not staged)
        if (i > 0) merge_pending(i - 1, 1);
      }
      if (n_pend > 0) merge_pending(n_pend - 1, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Per-device caches filled on first use (relaxed atomics: concurrent first
// calls store the same values).
std::atomic<bool> g_attr_set[4][64];  // [fp8 + 2 * fused][device]
std::atomic<int> g_num_sms[64];

}  // namespace

mla_status launch_decode(const DecodeLaunch &d, cudaStream_t stream, bool *merged) {
  *merged = false;
  const mla_decode_args &a = *d.a;
  const bool fp8 = a.kv_dtype == MLA_KV_FP8_E4M3;
  CUtensorMap tm_q, tm_kv;
  mla_status st = make_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 576,
                               static_cast<uint64_t>(a.num_rows) * a.num_heads, 64, kRows,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MLA_OK) return st;
  // page size >= 64: a tile is 64 rows of one sub-page, loaded as one 3-D
  // box of all nine chunks; smaller pages: one 2-D box per chunk and page.
  const bool tile3d = a.page_size >= kTileTok;
  const int box_rows = tile3d ? kTileTok : a.page_size;
  const CUtensorMapDataType kv_type = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle kv_swz = fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  if (tile3d)
    st = make_tmap_tile3d(&tm_kv, a.kv_cache, kv_type, fp8 ? 1 : 2, static_cast<uint64_t>(a.num_cache_rows),
                          box_rows, kv_swz);
  else
    st = make_tmap_2d(&tm_kv, a.kv_cache, kv_type, fp8 ? 1 : 2, 576, static_cast<uint64_t>(a.num_cache_rows), 64,
                      box_rows, kv_swz);
  if (st != MLA_OK) return st;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return MLA_ERR_CUDA;
  }
  // the in-kernel merge is its own instantiation: the default kernel holds none of its code
  const bool fuse_req = (a.flags & MLA_DECODE_FUSED_MERGE) != 0;
  auto kern = fp8 ? (fuse_req ? mla_decode_kernel<true, true> : mla_decode_kernel<true, false>)
                  : (fuse_req ? mla_decode_kernel<false, true> : mla_decode_kernel<false, false>);
  const int kind = (fp8 ? 1 : 0) + (fuse_req ? 2 : 0);
  if (!g_attr_set[kind][dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode smem)");
    g_attr_set[kind][dev].store(true, std::memory_order_relaxed);
  }
  int num_sms = g_num_sms[dev].load(std::memory_order_relaxed);
  if (num_sms == 0) {
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_num_sms[dev].store(num_sms, std::memory_order_relaxed);
  }

  Params p{};
  p.qo_indptr = a.qo_indptr;
  p.row_len = a.row_len;
  p.subpage_table = a.subpage_table;
  p.segm_out = reinterpret_cast<__nv_bfloat16 *>(d.segm_out);
  p.segm_max = d.segm_max;
  p.segm_sum = d.segm_sum;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.err = d.err;
  p.sched = d.sched;
  p.num_cache_rows = a.num_cache_rows;
  constexpr long long kDefaultBudget = 4000000000LL;  // ~2 s of SM clock
  p.wait_budget = a.wait_cycles > 0 ? static_cast<long long>(a.wait_cycles) : kDefaultBudget;
  p.drain_budget = kDefaultBudget;
  p.subpage_stride = a.subpage_stride;
  p.page_size = a.page_size;
  p.num_heads = a.num_heads;
  p.num_segments = a.num_segments;
  p.row_blocks = (a.max_qlen * a.num_heads + kRows - 1) / kRows;
  const int V = a.num_views > 1 ? a.num_views : 1;
  const int64_t items = static_cast<int64_t>(a.num_reqs) * V * p.row_blocks * a.num_segments;
  if (items > INT32_MAX) {
    set_error("mla_decode_verify: too many work items (%lld)", (long long)items);
    return MLA_ERR_UNSUPPORTED;
  }
  p.num_items = static_cast<int>(items);
  p.num_reqs = a.num_reqs;
  p.num_views = V;
  p.max_qlen = a.max_qlen;
  p.num_rows = a.num_rows;
  p.max_len = a.subpage_stride * a.page_size;
  p.tile3d = tile3d ? 1 : 0;
  const int64_t units = static_cast<int64_t>(a.num_reqs) * V * p.row_blocks;
  p.num_units = static_cast<int>(units);
  // the balanced split counts positions (tiles + one per unit) in int32:
  // every unit at the static bound must fit
  const int64_t max_unit_tiles = (static_cast<int64_t>(a.subpage_stride) * a.page_size + kTileTok - 1) / kTileTok;
  p.balanced = (a.num_segments >= 2 && (a.flags & MLA_DECODE_UNIFORM_SEGMENTS) == 0 && units <= kMaxUnits &&
                units * (max_unit_tiles + 1) <= INT32_MAX)
                   ? 1
                   : 0;
  p.unit_state = d.unit_state;
  p.fused = fuse_req ? 1 : 0;
  if (fuse_req && !p.balanced) {
    set_error("mla_decode_verify: MLA_DECODE_FUSED_MERGE needs the balanced split (num_segments > 1, "
              "at most %d units, no MLA_DECODE_UNIFORM_SEGMENTS)", kMaxUnits);
    return MLA_ERR_UNSUPPORTED;
  }
  *merged = fuse_req;
  const float kv_scale = fp8 ? a.kv_scale : 1.0f;
  p.score_scale_log2 = static_cast<float>(static_cast<double>(a.sm_scale) * kv_scale * 1.4426950408889634);
  p.out_scale = kv_scale;

  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  // The work counter and the unit counters are read only by the dynamic
  // schedule and by the in-kernel merge; the balanced split alone takes
  // chunk c on CTA c and needs neither.
  if (!p.balanced || p.fused) {
    e = cudaMemsetAsync(d.sched, 0, d.state_bytes, stream);  // work counter + unit counters
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(work counters)");
  }
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, stream, tm_q, tm_kv, p);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return MLA_OK;
}

}  // namespace mla
