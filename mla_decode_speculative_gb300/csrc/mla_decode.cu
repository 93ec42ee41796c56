// mla_decode.cu -- absorbed-form MLA decode / causal multi-token verify over a
// paged latent KV cache, one CTA per (request, 64-row block, split-K segment).
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
//  * The rows of a request (heads x qlen <= 64 per CTA) are processed jointly
//    against shared KV tiles of 128 tokens, so each latent row is read from
//    HBM once per request (the pages replicate the request per verify row).
//  * Swapped operand order, so every UMMA is M = 128 and the O accumulator
//    fits TMEM densely:
//        S^T[128 tok, 64 rows]   = K_tile[128, 576] . Q[64, 576]^T   (K-major A, K-major B)
//        O^T[4x128 dims, 64 rows] += V^T[512, 128 tok] . P^T[64, 128]^T (MN-major A, MN-major B)
//    TMEM: O^T in columns 0-255 (4 blocks x 64), S^T in columns 256-319.
//  * 8 shared-memory slots of 128 tokens x 64 dims (16 KB, 128-byte swizzle)
//    hold one tile: V chunk c always lives in slot c so PV operands are
//    adjacent; the rope chunk (dims 512-575) borrows slot 0 first and is
//    released as soon as its QK UMMAs finish.  Q (64 x 576) stays resident.
//  * Warp roles: warps 0-7 softmax (column group g = warp / 4 owns rows
//    32g..32g+31; TMEM lane quarter = warp % 4), warp 8 TMA producer, warp 9
//    UMMA issuer and TMEM owner.  fp8 tiles are TMA-loaded into the upper
//    half of a slot and expanded in place to bf16 by the softmax warps.
//  * Lazy rescaling: the running reference max only moves when a tile's max
//    exceeds it by more than 2^8, so O is rarely rescaled in TMEM.
//  * Every wait is bounded; a timeout records MLA_DEV_WAIT_TIMEOUT, lets all
//    roles drain without skipping a barrier, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mla_internal.h"
#include "mla_ptx.cuh"

namespace mla {
namespace {

constexpr int kTileTok = 128;      // KV tokens per tile (UMMA M of the QK product)
constexpr int kRows = 64;          // query rows per CTA (UMMA N)
constexpr int kNumChunks = 9;      // 576 / 64 dims per 128-byte swizzled chunk
constexpr int kRopeChunk = 8;      // dims 512..575
constexpr int kSlotBytes = kTileTok * 128;     // 16 KB
constexpr int kQChunkBytes = kRows * 128;      // 8 KB
constexpr int kPBytes = kTileTok * 128;        // P^T: [128 tokens][64 rows] bf16
constexpr int kNumSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

constexpr int kOffSlots = 0;
constexpr int kOffQ = kOffSlots + 8 * kSlotBytes;
constexpr int kOffP = kOffQ + kNumChunks * kQChunkBytes;
constexpr int kOffMisc = kOffP + kPBytes;

struct Misc {
  uint64_t full[8];
  uint64_t ready[8];  // fp8 only: slot expanded to bf16
  uint64_t empty[8];
  uint64_t q_full, s_full, p_full, o_done, fin;
  uint32_t tmem_base;
  int abort;
  alignas(16) int row_len[kRows];
  float red[2][2][4][32];  // [buffer][column group][lane quarter][lane]
};
constexpr int kSmemBytes = kOffMisc + static_cast<int>(sizeof(Misc)) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
  const int32_t *qo_indptr;
  const int32_t *row_len;
  const int32_t *subpage_table;
  float *segm_out;
  float *segm_max;
  float *segm_sum;
  __nv_bfloat16 *out;
  float *lse;
  int *err;
  int64_t num_cache_rows;
  long long wait_budget;
  int subpage_stride;
  int page_size;
  int num_heads;
  int num_segments;
  int max_qlen;
  int num_rows;
  int max_len;
  float score_scale_log2;  // sm_scale * kv_scale * log2(e)
  float out_scale;         // kv_scale (fp8) or 1
};

__device__ __forceinline__ void record_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Slot / chunk order of one tile's nine loads: the rope chunk first into
// slot 0, V chunks 1..7 into slots 1..7, then V chunk 0 into slot 0 again.
__device__ __forceinline__ int load_chunk(int li) { return li == 0 ? kRopeChunk : (li == 8 ? 0 : li); }
__device__ __forceinline__ int load_slot(int li) { return (li == 0 || li == 8) ? 0 : li; }
// Phase parity a consumer of load li of tile i waits for on full/ready[slot].
__device__ __forceinline__ uint32_t fill_parity(int li, int i) {
  return load_slot(li) == 0 ? (li == 0 ? 0u : 1u) : (static_cast<uint32_t>(i) & 1u);
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

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                      const Params p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the shared-window address (the 128-byte swizzle
  // pattern repeats every 1024 bytes and the descriptors assume that phase).
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc &misc = *reinterpret_cast<Misc *>(smem + kOffMisc);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t s_slots = s_base + kOffSlots;
  const uint32_t s_q = s_base + kOffQ;
  const uint32_t s_p = s_base + kOffP;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int rb = blockIdx.y;
  const int seg = blockIdx.x;
  const int H = p.num_heads;
  const int S = p.num_segments;
  const int P = p.page_size;

  // ---- work of this CTA (uniform over the CTA; exits happen before any barrier)
  const int q0 = p.qo_indptr[b];
  const int q1 = p.qo_indptr[b + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.num_rows || q1 - q0 > p.max_qlen) {
    if (threadIdx.x == 0 && rb == 0 && seg == 0) record_error(p.err, MLA_DEV_BAD_INDPTR);
    return;
  }
  const int rows_req = (q1 - q0) * H;
  const int row_begin = rb * kRows;
  if (row_begin >= rows_req) return;
  const int n_rows = min(kRows, rows_req - row_begin);
  const int row_base = q0 * H + row_begin;  // flattened (t, h) index of column 0

  int group_len = 0;  // longest row of the request: fixes the segment partition
  bool len_bad = false;
  for (int t = q0; t < q1; ++t) {
    int l = p.row_len[t];
    if (l > p.max_len) { len_bad = true; l = p.max_len; }
    group_len = max(group_len, max(l, 0));
  }
  if (len_bad && threadIdx.x == 0 && seg == 0) record_error(p.err, MLA_DEV_LEN_BOUND);
  const long long span = static_cast<long long>(S) * P;
  const int seg_tokens = static_cast<int>((group_len + span - 1) / span) * P;
  const int seg_lo = seg * seg_tokens;
  const int seg_hi = min(seg_lo + seg_tokens, group_len);
  const bool direct = (S == 1);

  if (seg_lo >= seg_hi) {
    // Nothing visible in this segment for any row of the block.
    for (int c = threadIdx.x; c < n_rows; c += kThreads) {
      const int64_t r = row_base + c;
      if (direct) p.lse[r] = -INFINITY;
      else { p.segm_max[r * S + seg] = -INFINITY; p.segm_sum[r * S + seg] = 0.0f; }
    }
    if (direct) {
      for (int e = threadIdx.x; e < n_rows * (512 / 8); e += kThreads) {
        const int64_t r = row_base + e / 64;
        reinterpret_cast<uint4 *>(p.out + r * 512)[e % 64] = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  const int n_tiles = (seg_hi - seg_lo + kTileTok - 1) / kTileTok;

  // ---- setup: TMEM, barriers, per-column lengths
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&misc.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_init(smem_u32(&misc.full[i]), 1);
      mbar_init(smem_u32(&misc.ready[i]), kNumSoftmaxWarps);
      mbar_init(smem_u32(&misc.empty[i]), 1);
    }
    mbar_init(smem_u32(&misc.q_full), 1);
    mbar_init(smem_u32(&misc.s_full), 1);
    mbar_init(smem_u32(&misc.p_full), kNumSoftmaxWarps);
    mbar_init(smem_u32(&misc.o_done), 1);
    mbar_init(smem_u32(&misc.fin), 1);
    misc.abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < kRows) {
    int l = 0;
    if (threadIdx.x < n_rows) {
      const int t = (row_begin + threadIdx.x) / H;
      l = min(max(p.row_len[q0 + t], 0), p.max_len);
    }
    misc.row_len[threadIdx.x] = l;
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
    // ======================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kv);
      const uint64_t pol_kv = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      const uint32_t q_bar = smem_u32(&misc.q_full);
      mbar_arrive_expect_tx(q_bar, kNumChunks * kQChunkBytes);
      for (int c = 0; c < kNumChunks; ++c)
        tma_load_2d(s_q + c * kQChunkBytes, &tm_q, q_bar, c * 64, row_base, pol_q);

      const int32_t *sp_row = p.subpage_table + static_cast<int64_t>(b) * p.subpage_stride;
      const int page_bytes = P * (kFp8 ? 64 : 128);
      // At most one load per slot can be in flight (a slot is refilled only
      // after its previous contents were consumed): remember the latest one.
      uint32_t armed = 0;          // slots that received a load
      uint32_t armed_par = 0;      // parity of that load's phase (bit per slot)
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int tok0 = seg_lo + i * kTileTok;
        const int n_valid = min(kTileTok, seg_hi - tok0);
        const int n_pages = (n_valid + P - 1) / P;
        int32_t rows_of_page[kTileTok / 8];
        for (int k = 0; k < n_pages; ++k) {
          const int32_t id = sp_row[tok0 / P + k];
          if (id < 0 || static_cast<int64_t>(id) * P + P > p.num_cache_rows) {
            record_error(p.err, MLA_DEV_BAD_SUBPAGE);
            rows_of_page[k] = static_cast<int32_t>(p.num_cache_rows);  // out of range: zero fill
          } else {
            rows_of_page[k] = id * P;
          }
        }
        for (int li = 0; li < kNumChunks; ++li) {
          const int c = load_chunk(li);
          const int sl = load_slot(li);
          const uint32_t wpar = fill_parity(li, i) ^ 1u;  // wait for the previous release
          if (!mbar_wait(smem_u32(&misc.empty[sl]), wpar, abort_flag, budget)) { fail(); ok = false; break; }
          const uint32_t fbar = smem_u32(&misc.full[sl]);
          mbar_arrive_expect_tx(fbar, n_pages * page_bytes);
          const uint32_t dst = s_slots + sl * kSlotBytes + (kFp8 ? kSlotBytes / 2 : 0);
          for (int k = 0; k < n_pages; ++k)
            tma_load_2d(dst + k * page_bytes, &tm_kv, fbar, c * 64, rows_of_page[k], pol_kv);
          armed |= 1u << sl;
          armed_par = (armed_par & ~(1u << sl)) | (fill_parity(li, i) << sl);
        }
      }
      if (!ok || *abort_flag) {
        // Let the copies already issued land before the CTA's memory is released.
        for (int sl = 0; sl < 8; ++sl)
          if (armed & (1u << sl)) {
            const volatile int never = 0;
            mbar_wait(smem_u32(&misc.full[sl]), (armed_par >> sl) & 1u, &never, budget);
          }
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================================================== UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kRows, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kRows, 1, 1);
      bool ok = mbar_wait(smem_u32(&misc.q_full), 0, abort_flag, budget);
      if (!ok) fail();
      tc_fence_after();
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int n_valid = min(kTileTok, seg_hi - (seg_lo + i * kTileTok));
        for (int li = 0; li < kNumChunks; ++li) {
          const int c = load_chunk(li);
          const int sl = load_slot(li);
          const uint32_t bar = smem_u32(kFp8 ? &misc.ready[sl] : &misc.full[sl]);
          if (!mbar_wait(bar, fill_parity(li, i), abort_flag, budget)) { fail(); ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = s_slots + sl * kSlotBytes;
          const uint32_t b0 = s_q + c * kQChunkBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ss(tmem + kTmemS, sdesc_sw128(a0 + kk * 32, 0, 1024),
                         sdesc_sw128(b0 + kk * 32, 0, 1024), idesc_qk, (li > 0 || kk > 0) ? 1u : 0u);
          if (li == 0) umma_commit(smem_u32(&misc.empty[0]));  // rope chunk done with slot 0
        }
        if (!ok) break;
        umma_commit(smem_u32(&misc.s_full));
        if (!mbar_wait(smem_u32(&misc.p_full), static_cast<uint32_t>(i) & 1u, abort_flag, budget)) {
          fail();
          break;
        }
        tc_fence_after();
        const int n_k16 = (n_valid + 15) / 16;
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          const uint32_t a0 = s_slots + (2 * blk) * kSlotBytes;
          for (int k = 0; k < n_k16; ++k)
            umma_bf16_ss(tmem + kTmemO + blk * kRows, sdesc_sw128(a0 + k * 2048, kSlotBytes, 1024),
                         sdesc_sw128(s_p + k * 2048, kPBytes, 1024), idesc_pv,
                         (i > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&misc.empty[2 * blk]));
          umma_commit(smem_u32(&misc.empty[2 * blk + 1]));
        }
        umma_commit(smem_u32(&misc.o_done));
      }
      umma_commit(smem_u32(&misc.fin));
      const volatile int never = 0;
      mbar_wait(smem_u32(&misc.fin), 0, &never, budget);
    }
  } else {
    // ======================================================== softmax warps
    const int g = warp >> 2;           // column group: rows 32g .. 32g+31 of the block
    const int wq = warp & 3;           // TMEM lane quarter
    const int tok = wq * 32 + lane;    // token row of S^T (and dim row of an O^T block)
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const int my_col = 32 * g + lane;  // column whose statistics this lane keeps
    float l_part[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) l_part[j] = 0.0f;
    float m_ref = -INFINITY;
    int red_buf = 0;
    bool ok = true;

    for (int i = 0; i < n_tiles; ++i) {
      const int tok0 = seg_lo + i * kTileTok;
      const int n_valid = min(kTileTok, seg_hi - tok0);

      if constexpr (kFp8) {
        // Expand this tile's nine fp8 chunks to bf16 in place, in load order.
        const int t2 = threadIdx.x >> 1;  // token row 0..127
        const int hf = threadIdx.x & 1;   // which 32 of the 64 dims
        for (int li = 0; li < kNumChunks; ++li) {
          const int sl = load_slot(li);
          if (ok && !mbar_wait(smem_u32(&misc.full[sl]), fill_parity(li, i), abort_flag, budget)) {
            fail();
            ok = false;
          }
          const uint32_t slot = s_slots + sl * kSlotBytes;
          const uint4 c0 = ld_shared_v4(slot + kSlotBytes / 2 + t2 * 64 + hf * 32);
          const uint4 c1 = ld_shared_v4(slot + kSlotBytes / 2 + t2 * 64 + hf * 32 + 16);
          named_bar_sync(3, kNumSoftmaxWarps * 32);
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t lo = w[2 * q], hi = w[2 * q + 1];
            const uint32_t chunk = static_cast<uint32_t>((hf * 4 + q) ^ (t2 & 7));
            st_shared_v4(slot + t2 * 128 + chunk * 16, e4m3x2_to_bf16x2(lo & 0xffff),
                         e4m3x2_to_bf16x2(lo >> 16), e4m3x2_to_bf16x2(hi & 0xffff),
                         e4m3x2_to_bf16x2(hi >> 16));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&misc.ready[sl]));
        }
      }

      if (ok && !mbar_wait(smem_u32(&misc.s_full), static_cast<uint32_t>(i) & 1u, abort_flag, budget)) {
        fail();
        ok = false;
      }
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_addr + kTmemS + 32 * g, sv);

      // scaled scores (log2 units), causal + segment mask per column
      float x[32];
      const int gtok = tok0 + tok;
      const bool tok_in = tok < n_valid;
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const int4 lens = *reinterpret_cast<const int4 *>(&misc.row_len[32 * g + 4 * j4]);
        const int lv[4] = {lens.x, lens.y, lens.z, lens.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = 4 * j4 + u;
          x[j] = (tok_in && gtok < lv[u]) ? __uint_as_float(sv[j]) * p.score_scale_log2 : -INFINITY;
        }
      }
      // column max over the 128 tokens of the tile
      float red[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) red[j] = x[j];
      const float wmax = warp_reduce_scatter<true>(red, lane);
      misc.red[red_buf][g][wq][lane] = wmax;
      named_bar_sync(1 + g, 128);
      const float tmax = fmaxf(fmaxf(misc.red[red_buf][g][0][lane], misc.red[red_buf][g][1][lane]),
                               fmaxf(misc.red[red_buf][g][2][lane], misc.red[red_buf][g][3][lane]));
      red_buf ^= 1;
      float alpha = 1.0f;
      if (tmax > m_ref + kRescaleThreshold) {
        alpha = exp2f(m_ref - tmax);  // 0 when m_ref is -inf
        m_ref = tmax;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
      const bool any_rescale = __any_sync(0xffffffffu, alpha != 1.0f);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float mj = __shfl_sync(0xffffffffu, m_use, j);
        x[j] = exp2f(x[j] - mj);  // probability (0 for masked entries)
      }
      if (any_rescale) {
#pragma unroll
        for (int j = 0; j < 32; ++j) l_part[j] *= __shfl_sync(0xffffffffu, alpha, j);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) l_part[j] += x[j];

      // PV of the previous tile must be done before P and O are touched.
      if (i > 0) {
        if (ok && !mbar_wait(smem_u32(&misc.o_done), static_cast<uint32_t>(i - 1) & 1u, abort_flag, budget)) {
          fail();
          ok = false;
        }
        tc_fence_after();
        if (any_rescale) {
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            const uint32_t taddr = tmem + lane_addr + kTmemO + blk * kRows + 32 * g;
            uint32_t ov[32];
            tmem_ld32(taddr, ov);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              ov[j] = __float_as_uint(__uint_as_float(ov[j]) * __shfl_sync(0xffffffffu, alpha, j));
            tmem_st32(taddr, ov);
          }
        }
      }
      // P^T row `tok`, columns 32g .. 32g+31 (bf16, 128-byte swizzle)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t chunk = static_cast<uint32_t>((4 * g + q) ^ (tok & 7));
        st_shared_v4(s_p + tok * 128 + chunk * 16, pack_bf16(x[8 * q + 0], x[8 * q + 1]),
                     pack_bf16(x[8 * q + 2], x[8 * q + 3]), pack_bf16(x[8 * q + 4], x[8 * q + 5]),
                     pack_bf16(x[8 * q + 6], x[8 * q + 7]));
      }
      // V rows past the last valid token but inside the last 16-token MMA step
      // hold stale or foreign data: zero them so 0 * V stays 0.
      if (!tok_in && tok < ((n_valid + 15) & ~15)) {
        for (int sl = 4 * g; sl < 4 * g + 4; ++sl)
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16)
            st_shared_v4(s_slots + sl * kSlotBytes + tok * 128 + c16 * 16, 0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&misc.p_full));
    }

    // ---- epilogue: row sums, statistics, output
    if (ok && !mbar_wait(smem_u32(&misc.o_done), static_cast<uint32_t>(n_tiles - 1) & 1u, abort_flag, budget)) {
      fail();
      ok = false;
    }
    tc_fence_after();
    const float wsum = warp_reduce_scatter<false>(l_part, lane);
    misc.red[red_buf][g][wq][lane] = wsum;
    named_bar_sync(1 + g, 128);
    const float l_tot = misc.red[red_buf][g][0][lane] + misc.red[red_buf][g][1][lane] +
                        misc.red[red_buf][g][2][lane] + misc.red[red_buf][g][3][lane];
    ok = ok && (*abort_flag == 0);
    if (ok && wq == 0 && my_col < n_rows) {
      const int64_t r = row_base + my_col;
      if (direct) {
        p.lse[r] = (l_tot > 0.0f) ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
      } else {
        p.segm_max[r * S + seg] = (l_tot > 0.0f) ? m_ref : -INFINITY;
        p.segm_sum[r * S + seg] = l_tot;
      }
    }
    const float col_scale = (l_tot > 0.0f) ? (direct ? p.out_scale / l_tot : p.out_scale) : 0.0f;
    const int n_cols = min(32, n_rows - 32 * g);
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t ov[32];
      tmem_ld32(tmem + lane_addr + kTmemO + blk * kRows + 32 * g, ov);
      if (!ok) continue;
      const int dim = blk * 128 + tok;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float sc = __shfl_sync(0xffffffffu, col_scale, j);
        const float lj = __shfl_sync(0xffffffffu, l_tot, j);
        if (j < n_cols) {
          const int64_t r = row_base + 32 * g + j;
          const float v = __uint_as_float(ov[j]) * sc;
          if (direct) p.out[r * 512 + dim] = __float2bfloat16_rn(v);
          else if (lj > 0.0f) p.segm_out[(r * S + seg) * 512 + dim] = v;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool g_attr_set[2][64];

}  // namespace

mla_status launch_decode(const DecodeLaunch &d, cudaStream_t stream) {
  const mla_decode_args &a = *d.a;
  const bool fp8 = a.kv_dtype == MLA_KV_FP8_E4M3;
  CUtensorMap tm_q, tm_kv;
  mla_status st = make_tmap_2d(&tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 576,
                               static_cast<uint64_t>(a.num_rows) * a.num_heads, 64, kRows,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MLA_OK) return st;
  if (fp8)
    st = make_tmap_2d(&tm_kv, a.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 576,
                      static_cast<uint64_t>(a.num_cache_rows), 64, a.page_size,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    st = make_tmap_2d(&tm_kv, a.kv_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 576,
                      static_cast<uint64_t>(a.num_cache_rows), 64, a.page_size,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MLA_OK) return st;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  auto kern = fp8 ? mla_decode_kernel<true> : mla_decode_kernel<false>;
  if (dev < 64 && !g_attr_set[fp8][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode smem)");
    g_attr_set[fp8][dev] = true;
  }

  Params p{};
  p.qo_indptr = a.qo_indptr;
  p.row_len = a.row_len;
  p.subpage_table = a.subpage_table;
  p.segm_out = d.segm_out;
  p.segm_max = d.segm_max;
  p.segm_sum = d.segm_sum;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.lse = a.lse;
  p.err = d.err;
  p.num_cache_rows = a.num_cache_rows;
  p.wait_budget = 4000000000LL;  // ~2 s of SM clock
  p.subpage_stride = a.subpage_stride;
  p.page_size = a.page_size;
  p.num_heads = a.num_heads;
  p.num_segments = a.num_segments;
  p.max_qlen = a.max_qlen;
  p.num_rows = a.num_rows;
  p.max_len = a.subpage_stride * a.page_size;
  const float kv_scale = fp8 ? a.kv_scale : 1.0f;
  p.score_scale_log2 = static_cast<float>(static_cast<double>(a.sm_scale) * kv_scale * 1.4426950408889634);
  p.out_scale = kv_scale;

  const int row_blocks = (a.max_qlen * a.num_heads + kRows - 1) / kRows;
  dim3 grid(a.num_segments, row_blocks, a.num_reqs);
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tm_q, tm_kv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return MLA_OK;
}

}  // namespace mla
