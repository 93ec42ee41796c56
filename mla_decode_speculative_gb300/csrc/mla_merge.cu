// mla_merge.cu -- merge of partial attention states into a bf16 output and a
// float32 natural-log LSE.
//
// Segment mode (vLLM #51705 digest, 实现拆解 4, merge_mla_segments_triton):
// S split-K partials per (row, head) in base 2 -- max m_s, exp2 sum l_s and
// unnormalised output acc_s -- are combined as
//   M = max m_s, c_s = 2^(m_s - M), out = sum c_s acc_s / sum c_s l_s,
//   lse = (M + log2 sum c_s l_s) * ln 2.
// State mode (vLLM #51705, 功能与动机; sglang #34432, merge_state_triton and
// 评论区精华 4): W normalised shard states (out_r, lse_r) in base e:
//   M = max lse_r, w_r = e^(lse_r - M), out = sum w_r out_r / sum w_r,
//   lse = M + ln sum w_r.
// An empty part (max / lse = -inf) contributes nothing; all parts empty
// gives out = 0, lse = -inf.
//
// Segment partials come in the decode kernel's block layout: per (request,
// 64-row block, segment) a bf16 block [8 row octets][512 dims][8 rows].  One
// CTA merges one row octet of one row block: every part's octet is one
// contiguous 8 KB run, streamed through a per-thread cp.async ring in shared
// memory (thread t: dims 2t, 2t + 1 of the 8 rows), with each row's
// statistics read once.  State partials are row-major [W][T*H][512] bf16: one
// warp per (row, head), lane l owning dims 16l .. 16l + 15.  Both are HBM/L2
// streaming reductions.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreadsPerItem = 128;  // state mode: 512 dims / 4 per thread
constexpr int kBlockRows = 64;        // segment mode: rows per partial block
constexpr float kLn2 = 0.69314718055994530942f;

struct StateParams {
  const __nv_bfloat16 *part_out;
  const float *part_lse;
  __nv_bfloat16 *out;
  float *lse;
  int64_t num_items;  // rows * heads
  int num_parts;
};

struct SegParams {
  const __nv_bfloat16 *segm_out;  // [B, RB, S, 8, 512, 8]
  const float *segm_max;          // [T*H, S]
  const float *segm_sum;
  const int32_t *qo_indptr;
  __nv_bfloat16 *out;
  float *lse;
  int num_rows;
  int num_heads;
  int num_parts;
  int row_blocks;
  int num_reqs;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ---------------------------------------------------------------- segments
constexpr int kSegChunk = 32;  // segments whose weights are staged at a time

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *gptr) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kOctSlot = 8 * 1024;  // one part's octet: [512 dims][8 rows] bf16
// Two shapes of the segment merge: a deep ring (8 slots, 3 CTAs per SM) for
// grids of up to two waves -- few units, each with many parts to stream --
// and a shallower ring at higher occupancy (6 slots, 4 CTAs per SM, <= 64
// registers) for larger grids, where resident CTAs count more than parts in
// flight (the bandwidth-sized merge: 0.82 -> 0.85 of measured HBM).
constexpr int kOctRingDeep = 8, kOctCtasDeep = 3;
constexpr int kOctRingWide = 6, kOctCtasWide = 4;

// grid (V * B * RB * 8), 256 threads: one (view, request, row block) unit x
// one row octet (8 rows).  Warp r takes the statistics of row r of the octet:
// its lanes the segments (32 at a time), warp reductions give the row's max
// and denominator; the normalised weights 2^(m_s - M) / den of 32 segments at
// a time go to shared memory and the segments with a weight for any of the 8
// rows are listed.  A part's octet is one contiguous 8 KB run of its block
// ([512 dims][8 rows]); thread t sums dims 2t and 2t + 1 for the 8 rows,
// streaming its two 16-byte pieces of every listed part through its own
// places in a kOctRing-deep shared-memory ring with cp.async (a commit group
// per part, up to kOctRing - 1 parts in flight, no registers held and, since
// a thread reads back only what it copied, no barrier inside the stream).
// The first two segments are copied before the statistics are known (a
// request's first segments hold its tokens; one that turns out empty just
// gets weight 0, which selects 0), so that their round trip overlaps the
// statistics'.  Each output row leaves as 128-byte warp stores.
template <int kOctRing, int kOctCtas>
__global__ void __launch_bounds__(256, kOctCtas) merge_segment_octets(const SegParams p) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ __align__(128) uint8_t ring[];  // [kOctRing][256 threads][2] x 16 B
  __shared__ __align__(16) float s_w[kSegChunk][8];
  __shared__ float s_M[8], s_inv[8];
  __shared__ int s_live[kSegChunk], s_list[kSegChunk], s_nlive;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = blockIdx.x >> 3, oct = blockIdx.x & 7;
  // unit (view, request, row block): vb = v * B + b
  const int vb = unit / p.row_blocks, rb = unit % p.row_blocks;
  const int v = vb / p.num_reqs, b = vb % p.num_reqs;
  const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.num_rows) return;  // flagged by the decode kernel
  const int rows_req = (q1 - q0) * p.num_heads;
  const int n_rows = min(8, rows_req - rb * kBlockRows - 8 * oct);  // rows of this octet
  if (n_rows <= 0) return;
  const int S = p.num_parts;
  const int64_t grow0 = (static_cast<int64_t>(v) * p.num_rows + q0) * p.num_heads + rb * kBlockRows + 8 * oct;
  const float *mx = p.segm_max + grow0 * S;  // [8 rows][S], contiguous
  const float *sm = p.segm_sum + grow0 * S;
  const int64_t blk0 = (static_cast<int64_t>(vb) * p.row_blocks + rb) * S;
  const uint32_t s_ring = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
  // this thread's pieces (dims 2 tid and 2 tid + 1, 8 rows each) of part `sc` into ring slot `slot`
  auto issue = [&](int sc, int slot) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p.segm_out + (blk0 + sc) * (512 * kBlockRows)) + oct * 512 + 2 * tid;
    const uint32_t dst = s_ring + slot * kOctSlot + tid * 32;
    cp_async16(dst, src);
    cp_async16(dst + 16, src + 1);
  };
  constexpr int kPre = 2;
  const int n_pre = min(kPre, S);
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    if (i < n_pre) issue(i, i);
    cp_async_commit();
  }
  // row statistics: warp r, lanes over the segments, a running (max, sum)
  {
    float M = -INFINITY, d = 0.0f;
    if (warp < n_rows) {
      for (int s0 = 0; s0 < S; s0 += 32) {
        const int s2 = s0 + lane;
        const float m = s2 < S ? mx[warp * S + s2] : -INFINITY;
        const float l = s2 < S ? sm[warp * S + s2] : 0.0f;
        const float nM = fmaxf(M, warp_max(m));
        if (nM != -INFINITY) {
          const float part = warp_sum(m != -INFINITY ? exp2f(m - nM) * l : 0.0f);
          d = (M != -INFINITY ? d * exp2f(M - nM) : 0.0f) + part;
          M = nM;
        }
      }
    }
    if (lane == 0) {
      s_M[warp] = M;
      s_inv[warp] = d > 0.0f ? 1.0f / d : 0.0f;
      if (warp < n_rows) p.lse[grow0 + warp] = d > 0.0f ? (M + log2f(d)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();

  float a[16];  // a[2 r]: row r, dim 2 tid;  a[2 r + 1]: row r, dim 2 tid + 1
#pragma unroll
  for (int k = 0; k < 16; ++k) a[k] = 0.0f;
  for (int c0 = 0; c0 < S; c0 += kSegChunk) {
    const int nc = min(kSegChunk, S - c0);
    const int pre = c0 == 0 ? n_pre : 0;  // slots already in the ring, live or not
    if (tid < kSegChunk) s_live[tid] = tid < pre ? 1 : 0;
    __syncthreads();
    {  // weights of this chunk: thread (slot tid / 8, row tid % 8)
      const int sc = tid >> 3, r = tid & 7;
      float w = 0.0f;
      if (sc < nc && r < n_rows && s_M[r] != -INFINITY) {
        const float m = mx[r * S + c0 + sc];
        if (m != -INFINITY) w = exp2f(m - s_M[r]) * s_inv[r];
      }
      s_w[sc][r] = w;
      if (w != 0.0f) s_live[sc] = 1;
    }
    __syncthreads();
    if (warp == 0) {  // the slots to sum, in order: the prefetched ones, then the live ones
      const bool lv = lane < nc && s_live[lane] != 0;
      const unsigned mk = __ballot_sync(0xffffffffu, lv);
      if (lv) s_list[__popc(mk & ((1u << lane) - 1u))] = lane;
      if (lane == 0) s_nlive = __popc(mk);
    }
    __syncthreads();
    const int n_live = s_nlive;
    // ring: parts i .. i + kOctRing - 2 in flight while part i is summed (the
    // first chunk's prefetched parts are ring slots 0 .. kPre - 1)
#pragma unroll
    for (int i = 0; i < kOctRing - 1; ++i) {
      if (c0 == 0 && i < kPre) continue;
      if (i < n_live) issue(c0 + s_list[i], i);
      cp_async_commit();
    }
    for (int i = 0; i < n_live; ++i) {
      if (i + kOctRing - 1 < n_live) issue(c0 + s_list[i + kOctRing - 1], (i + kOctRing - 1) % kOctRing);
      cp_async_commit();
      cp_async_wait<kOctRing - 1>();  // this thread's pieces of part i have landed
      const uint4 *slot = reinterpret_cast<const uint4 *>(ring + (i % kOctRing) * kOctSlot) + 2 * tid;
      const uint4 x0 = slot[0], x1 = slot[1];
      const int sc = s_list[i];
      const float4 wa = *reinterpret_cast<const float4 *>(&s_w[sc][0]);
      const float4 wb = *reinterpret_cast<const float4 *>(&s_w[sc][4]);
      const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      const uint32_t u0[4] = {x0.x, x0.y, x0.z, x0.w};  // dim 2 tid, rows 0..7
      const uint32_t u1[4] = {x1.x, x1.y, x1.z, x1.w};  // dim 2 tid + 1
#pragma unroll
      for (int r = 0; r < 8; ++r) {  // a weight of 0 selects 0: an empty row's slot is never a value
        const float e0 = (r & 1) ? bf16_hi(u0[r >> 1]) : bf16_lo(u0[r >> 1]);
        const float e1 = (r & 1) ? bf16_hi(u1[r >> 1]) : bf16_lo(u1[r >> 1]);
        a[2 * r] += (w[r] != 0.0f) ? w[r] * e0 : 0.0f;
        a[2 * r + 1] += (w[r] != 0.0f) ? w[r] * e1 : 0.0f;
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // s_w / s_live / s_list are refilled by the next chunk
  }
  // row r: dims 2 tid, 2 tid + 1 as one 4-byte store; a warp covers 128 bytes of the row
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < n_rows)
      reinterpret_cast<uint32_t *>(p.out + (grow0 + r) * 512)[tid] = pack_bf16(a[2 * r], a[2 * r + 1]);
}

// ---------------------------------------------------------------- states
constexpr int kStateWarps = 4;  // (row, head) items per 128-thread CTA, one per warp
constexpr int kStateBatch = 8;  // parts read at a time

// Up to 32 parts: one warp per (row, head).  Lane s holds part s's LSE; lane
// l covers dims 16 l .. 16 l + 15 of every part (two 16-byte loads per part,
// a warp's load covering the part's 1 KiB row whole).  The first eight parts'
// rows are read together with the LSEs (one round trip for up to eight
// shards); a part with lse = -inf gets weight 0, which selects 0, so its row
// is never used as a value.
__global__ void __launch_bounds__(kStateWarps * 32) merge_states_small(const StateParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int64_t it = static_cast<int64_t>(blockIdx.x) * kStateWarps + (threadIdx.x >> 5);
  if (it >= p.num_items) return;
  const int n = p.num_parts;
  auto row_of = [&](int s) {
    return reinterpret_cast<const uint4 *>(p.part_out + (static_cast<int64_t>(s) * p.num_items + it) * 512) + 2 * lane;
  };
  uint4 x[kStateBatch][2];
#pragma unroll
  for (int u = 0; u < kStateBatch; ++u) {
    if (u < n) {
      x[u][0] = __ldcs(row_of(u));
      x[u][1] = __ldcs(row_of(u) + 1);
    }
  }
  const float m = lane < n ? p.part_lse[static_cast<int64_t>(lane) * p.num_items + it] : -INFINITY;
  const float M = warp_max(m);
  uint4 *dst = reinterpret_cast<uint4 *>(p.out + it * 512) + 2 * lane;
  if (M == -INFINITY) {
    dst[0] = dst[1] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) p.lse[it] = -INFINITY;
    return;
  }
  const float w = (m != -INFINITY) ? expf(m - M) : 0.0f;
  const float den = warp_sum(w);
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
  for (int s0 = 0; s0 < n; s0 += kStateBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int u = 0; u < kStateBatch; ++u) {
        if (s0 + u < n) {
          x[u][0] = __ldcs(row_of(s0 + u));
          x[u][1] = __ldcs(row_of(s0 + u) + 1);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kStateBatch; ++u) {
      const float ws = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);
      if (s0 + u >= n || ws == 0.0f) continue;
      const uint32_t vv[8] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w,
                              x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[2 * k] = fmaf(ws, bf16_lo(vv[k]), acc[2 * k]);
        acc[2 * k + 1] = fmaf(ws, bf16_hi(vv[k]), acc[2 * k + 1]);
      }
    }
  }
  const float inv_den = 1.0f / den;
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = pack_bf16(acc[2 * k] * inv_den, acc[2 * k + 1] * inv_den);
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  if (lane == 0) p.lse[it] = M + logf(den);
}

__device__ __forceinline__ float4 load_state4(const StateParams &p, int64_t it, int s, int tid) {
  const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(
                             p.part_out + (static_cast<int64_t>(s) * p.num_items + it) * 512) + tid);
  return make_float4(bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y));
}

// Any number of parts: live parts are compacted, in order, into shared
// memory, then streamed with eight loads in flight per thread.
__global__ void __launch_bounds__(kThreadsPerItem) merge_states(const StateParams p) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float s_w[kMaxParts];
  __shared__ int s_idx[kMaxParts];
  __shared__ float s_red[kThreadsPerItem / 32];
  __shared__ int s_cnt[kThreadsPerItem / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t it = blockIdx.x;
  const int n = p.num_parts;
  auto stat = [&](int s) -> float { return p.part_lse[static_cast<int64_t>(s) * p.num_items + it]; };
  float m_loc = -INFINITY;
  for (int s = tid; s < n; s += kThreadsPerItem) m_loc = fmaxf(m_loc, stat(s));
  m_loc = warp_max(m_loc);
  if (lane == 0) s_red[warp] = m_loc;
  __syncthreads();
  float M = s_red[0];
#pragma unroll
  for (int k = 1; k < kThreadsPerItem / 32; ++k) M = fmaxf(M, s_red[k]);
  __syncthreads();
  uint2 *dst = reinterpret_cast<uint2 *>(p.out + it * 512) + tid;
  if (M == -INFINITY) {
    *dst = make_uint2(0, 0);
    if (tid == 0) p.lse[it] = -INFINITY;
    return;
  }
  float d_loc = 0.0f;
  int n_live = 0;
  for (int base = 0; base < n; base += kThreadsPerItem) {
    const int s = base + tid;
    float wgt = 0.0f;
    if (s < n) {
      const float m = stat(s);
      if (m != -INFINITY) {
        wgt = expf(m - M);
        d_loc += wgt;
      }
    }
    const unsigned live = __ballot_sync(0xffffffffu, wgt != 0.0f);
    if (lane == 0) s_cnt[warp] = __popc(live);
    __syncthreads();
    int off = n_live;
    for (int k = 0; k < warp; ++k) off += s_cnt[k];
    if (wgt != 0.0f) {
      const int pos = off + __popc(live & ((1u << lane) - 1u));
      s_w[pos] = wgt;
      s_idx[pos] = s;
    }
    for (int k = 0; k < kThreadsPerItem / 32; ++k) n_live += s_cnt[k];
    __syncthreads();
  }
  d_loc = warp_sum(d_loc);
  if (lane == 0) s_red[warp] = d_loc;
  __syncthreads();
  float den = 0.0f;
#pragma unroll
  for (int k = 0; k < kThreadsPerItem / 32; ++k) den += s_red[k];
  const float inv_den = 1.0f / den;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int k0 = 0; k0 < n_live; k0 += 8) {
    float4 v[8];
    float wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = min(k0 + u, n_live - 1);  // padding re-reads the last live part, weight 0
      wv[u] = (k0 + u < n_live) ? s_w[k] : 0.0f;
      v[u] = load_state4(p, it, s_idx[k], tid);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc[0] = fmaf(wv[u], v[u].x, acc[0]);
      acc[1] = fmaf(wv[u], v[u].y, acc[1]);
      acc[2] = fmaf(wv[u], v[u].z, acc[2]);
      acc[3] = fmaf(wv[u], v[u].w, acc[3]);
    }
  }
  *dst = make_uint2(pack_bf16(acc[0] * inv_den, acc[1] * inv_den),
                    pack_bf16(acc[2] * inv_den, acc[3] * inv_den));
  if (tid == 0) p.lse[it] = M + logf(den);
}

// Per device: the segment merge's shared-memory attribute is set (relaxed
// atomics: concurrent first calls store the same value).
std::atomic<bool> g_seg_attr_set[2][64];  // [shape][device]
std::atomic<int> g_seg_sms[64];

}  // namespace

mla_status launch_merge(const MergeLaunch &m, cudaStream_t stream) {
  if (m.mode == MLA_MERGE_SEGMENTS) {
    if (m.num_reqs == 0 || m.num_rows == 0) return MLA_OK;
    SegParams p{};
    p.segm_out = reinterpret_cast<const __nv_bfloat16 *>(m.segm_out);
    p.segm_max = m.segm_max;
    p.segm_sum = m.segm_sum;
    p.qo_indptr = m.qo_indptr;
    p.out = static_cast<__nv_bfloat16 *>(m.out);
    p.lse = m.lse;
    p.num_rows = m.num_rows;
    p.num_heads = m.num_heads;
    p.num_parts = m.num_parts;
    p.row_blocks = m.row_blocks;
    p.num_reqs = m.num_reqs;
    const int64_t ctas = static_cast<int64_t>(m.num_reqs) * m.num_views * m.row_blocks;
    if (ctas > INT32_MAX || m.row_blocks < 1) {
      set_error("mla_merge_segments: bad row-block count (%lld)", (long long)ctas);
      return MLA_ERR_UNSUPPORTED;
    }
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return cuda_fail(e0, "merge: device");
    if (dev < 0 || dev >= 64) {
      set_error("device ordinal %d out of range", dev);
      return MLA_ERR_CUDA;
    }
    int sms = g_seg_sms[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
      e0 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e0 != cudaSuccess) return cuda_fail(e0, "cudaDeviceGetAttribute(SM count)");
      g_seg_sms[dev].store(sms, std::memory_order_relaxed);
    }
    // more than two waves at the deep shape's occupancy: take the wide shape
    const bool wide = ctas * 8 > 2 * static_cast<int64_t>(kOctCtasDeep) * sms;
    auto kern = wide ? merge_segment_octets<kOctRingWide, kOctCtasWide> : merge_segment_octets<kOctRingDeep, kOctCtasDeep>;
    const int dyn = (wide ? kOctRingWide : kOctRingDeep) * kOctSlot;
    if (!g_seg_attr_set[wide][dev].load(std::memory_order_relaxed)) {
      e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
      if (e0 != cudaSuccess) return cuda_fail(e0, "cudaFuncSetAttribute(merge smem)");
      g_seg_attr_set[wide][dev].store(true, std::memory_order_relaxed);
    }
    if (ctas * 8 > INT32_MAX) {
      set_error("mla_merge_segments: too many row blocks (%lld)", (long long)ctas);
      return MLA_ERR_UNSUPPORTED;
    }
    const cudaError_t el = launch_pdl(kern, dim3(static_cast<unsigned>(ctas * 8)), dim3(256), dyn, stream, p);
    if (el != cudaSuccess) return cuda_fail(el, "merge launch");
  } else {
    StateParams p{};
    p.part_out = static_cast<const __nv_bfloat16 *>(m.part_out);
    p.part_lse = m.part_lse;
    p.out = static_cast<__nv_bfloat16 *>(m.out);
    p.lse = m.lse;
    p.num_items = static_cast<int64_t>(m.num_rows) * m.num_heads;
    p.num_parts = m.num_parts;
    if (p.num_items == 0) return MLA_OK;
    if (p.num_items > INT32_MAX) {
      set_error("mla_merge_segments: too many (row, head) items");
      return MLA_ERR_UNSUPPORTED;
    }
    const unsigned blocks = static_cast<unsigned>(p.num_items);
    if (p.num_parts <= 32) {
      const unsigned ctas = static_cast<unsigned>((p.num_items + kStateWarps - 1) / kStateWarps);
      const cudaError_t el = launch_pdl(merge_states_small, dim3(ctas), dim3(kStateWarps * 32), 0, stream, p);
      if (el != cudaSuccess) return cuda_fail(el, "merge launch");
    } else {
      const cudaError_t el = launch_pdl(merge_states, dim3(blocks), dim3(kThreadsPerItem), 0, stream, p);
      if (el != cudaSuccess) return cuda_fail(el, "merge launch");
    }
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return MLA_OK;
}

}  // namespace mla
