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
// An empty part (max / lse = -inf) is never read; all parts empty gives
// out = 0, lse = -inf.
//
// Both modes read bf16 partial outputs (segment partials are stored in bf16
// by the decode kernel).  HBM-bound streaming reduction: one 128-thread
// block per (row, head); each thread owns 4 of the 512 output dims, reads
// each live part with one 8-byte streaming load (8 parts in flight per
// thread) and writes 8 bytes of bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreadsPerItem = 128;  // 512 dims / 4 per thread
constexpr float kLn2 = 0.69314718055994530942f;

struct MergeParams {
  const __nv_bfloat16 *segm_out;
  const float *segm_max;
  const float *segm_sum;
  const __nv_bfloat16 *part_out;
  const float *part_lse;
  __nv_bfloat16 *out;
  float *lse;
  const int32_t *live_rows;
  int64_t num_items;  // rows * heads
  int num_heads;
  int num_parts;
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
// Loads this thread's 4 dims of part s of item it.
template <bool kSeg>
__device__ __forceinline__ float4 load4(const MergeParams &p, int64_t it, int s, int tid) {
  const __nv_bfloat16 *src = kSeg ? p.segm_out + (it * p.num_parts + s) * 512
                                  : p.part_out + (static_cast<int64_t>(s) * p.num_items + it) * 512;
  const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(src) + tid);
  return make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u),
                     __uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
}

// Up to 32 parts: no block barrier.  Every thread reads the item's (tiny,
// L1-broadcast) statistics itself, so the loads of all live parts are issued
// together, one dependent round trip after the statistics.
template <bool kSeg>
__global__ void __launch_bounds__(kThreadsPerItem) merge_kernel_small(const MergeParams p) {
  const int tid = threadIdx.x;
  const int64_t it = blockIdx.x;
  if (p.live_rows != nullptr && it / p.num_heads >= static_cast<int64_t>(*p.live_rows)) return;
  const int n = p.num_parts;
  float m[32], l[32];
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    m[s] = -INFINITY;
    l[s] = 0.0f;
    if (s < n) {
      if constexpr (kSeg) {
        m[s] = p.segm_max[it * n + s];
        l[s] = p.segm_sum[it * n + s];
      } else {
        m[s] = p.part_lse[static_cast<int64_t>(s) * p.num_items + it];
      }
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < 32; ++s) M = fmaxf(M, m[s]);
  uint2 *dst = reinterpret_cast<uint2 *>(p.out + it * 512) + tid;
  if (M == -INFINITY) {
    *dst = make_uint2(0, 0);
    if (tid == 0) p.lse[it] = -INFINITY;
    return;
  }
  float den = 0.0f;
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    float w = 0.0f;
    if (m[s] != -INFINITY) w = kSeg ? exp2f(m[s] - M) : expf(m[s] - M);
    den += kSeg ? w * l[s] : w;
    m[s] = w;  // m now holds the weights
  }
  float4 v[32];
#pragma unroll
  for (int s = 0; s < 32; ++s)
    v[s] = (m[s] != 0.0f) ? load4<kSeg>(p, it, s, tid) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    acc[0] = fmaf(m[s], v[s].x, acc[0]);
    acc[1] = fmaf(m[s], v[s].y, acc[1]);
    acc[2] = fmaf(m[s], v[s].z, acc[2]);
    acc[3] = fmaf(m[s], v[s].w, acc[3]);
  }
  const float inv_den = 1.0f / den;
  *dst = make_uint2(pack_bf16(acc[0] * inv_den, acc[1] * inv_den),
                    pack_bf16(acc[2] * inv_den, acc[3] * inv_den));
  if (tid == 0) p.lse[it] = kSeg ? (M + log2f(den)) * kLn2 : M + logf(den);
}

// One 128-thread block per (row, head): thread t owns output dims 4t..4t+3,
// so every live part costs each thread one 8-byte load, and up to 8 parts
// are in flight per thread.
template <bool kSeg>
__global__ void __launch_bounds__(kThreadsPerItem) merge_kernel(const MergeParams p) {
  __shared__ float s_w[kMaxParts];
  __shared__ int s_idx[kMaxParts];
  __shared__ float s_red[kThreadsPerItem / 32];
  __shared__ int s_cnt[kThreadsPerItem / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t it = blockIdx.x;
  if (p.live_rows != nullptr && it / p.num_heads >= static_cast<int64_t>(*p.live_rows)) return;
  const int n = p.num_parts;

  // statistic of part s: base-2 max (segments) or natural-log lse (states)
  auto stat = [&](int s) -> float {
    if constexpr (kSeg) return p.segm_max[it * n + s];
    else return p.part_lse[static_cast<int64_t>(s) * p.num_items + it];
  };
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
  // unnormalised weights and the denominator; live parts are compacted, in
  // order, into (s_idx, s_w) so the load loop below has no conditionals
  float d_loc = 0.0f;
  int n_live = 0;
  for (int base = 0; base < n; base += kThreadsPerItem) {
    const int s = base + tid;
    float wgt = 0.0f;
    if (s < n) {
      const float m = stat(s);
      if (m != -INFINITY) {
        if constexpr (kSeg) {
          wgt = exp2f(m - M);
          d_loc += wgt * p.segm_sum[it * n + s];
        } else {
          wgt = expf(m - M);
          d_loc += wgt;
        }
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
    float v[8][4];
    float wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = min(k0 + u, n_live - 1);  // padding re-reads the last live part, weight 0
      const int s = s_idx[k];
      wv[u] = (k0 + u < n_live) ? s_w[k] : 0.0f;
      const __nv_bfloat16 *src = kSeg ? p.segm_out + (it * n + s) * 512
                                      : p.part_out + (static_cast<int64_t>(s) * p.num_items + it) * 512;
      const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(src) + tid);
      v[u][0] = __uint_as_float(x.x << 16);
      v[u][1] = __uint_as_float(x.x & 0xffff0000u);
      v[u][2] = __uint_as_float(x.y << 16);
      v[u][3] = __uint_as_float(x.y & 0xffff0000u);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = fmaf(wv[u], v[u][c], acc[c]);
  }
  *dst = make_uint2(pack_bf16(acc[0] * inv_den, acc[1] * inv_den),
                    pack_bf16(acc[2] * inv_den, acc[3] * inv_den));
  if (tid == 0) p.lse[it] = kSeg ? (M + log2f(den)) * kLn2 : M + logf(den);
}

}  // namespace

mla_status launch_merge(const MergeLaunch &m, cudaStream_t stream) {
  MergeParams p{};
  p.segm_out = reinterpret_cast<const __nv_bfloat16 *>(m.segm_out);
  p.segm_max = m.segm_max;
  p.segm_sum = m.segm_sum;
  p.part_out = static_cast<const __nv_bfloat16 *>(m.part_out);
  p.part_lse = m.part_lse;
  p.out = static_cast<__nv_bfloat16 *>(m.out);
  p.lse = m.lse;
  p.live_rows = m.live_rows;
  p.num_items = static_cast<int64_t>(m.num_rows) * m.num_heads;
  p.num_heads = m.num_heads;
  p.num_parts = m.num_parts;
  if (p.num_items == 0) return MLA_OK;
  if (p.num_items > INT32_MAX) {
    set_error("mla_merge_segments: too many (row, head) items");
    return MLA_ERR_UNSUPPORTED;
  }
  const unsigned blocks = static_cast<unsigned>(p.num_items);
  const bool small = p.num_parts <= 32;
  if (m.mode == MLA_MERGE_SEGMENTS) {
    if (small) merge_kernel_small<true><<<blocks, kThreadsPerItem, 0, stream>>>(p);
    else merge_kernel<true><<<blocks, kThreadsPerItem, 0, stream>>>(p);
  } else {
    if (small) merge_kernel_small<false><<<blocks, kThreadsPerItem, 0, stream>>>(p);
    else merge_kernel<false><<<blocks, kThreadsPerItem, 0, stream>>>(p);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return MLA_OK;
}

}  // namespace mla
