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
// HBM-bound streaming reduction: one warp per (row, head); each lane owns 16
// of the 512 output dims, reads each live part with 16-byte streaming loads
// (4 parts in flight per lane) and writes 32 contiguous bytes of bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLn2 = 0.69314718055994530942f;

struct MergeParams {
  const float *segm_out;
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
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// Loads this lane's 16 dims of part `s` of item `it`.
template <bool kSeg>
__device__ __forceinline__ void load_part(const MergeParams &p, int64_t it, int s, int lane, float *v) {
  if constexpr (kSeg) {
    const float4 *src = reinterpret_cast<const float4 *>(
        p.segm_out + (it * p.num_parts + s) * 512 + lane * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 x = __ldcs(src + k);
      v[4 * k + 0] = x.x;
      v[4 * k + 1] = x.y;
      v[4 * k + 2] = x.z;
      v[4 * k + 3] = x.w;
    }
  } else {
    const uint4 *src = reinterpret_cast<const uint4 *>(
        p.part_out + (static_cast<int64_t>(s) * p.num_items + it) * 512 + lane * 16);
    const uint4 a = __ldcs(src);
    const uint4 b = __ldcs(src + 1);
    bf16x8_to_f32(a, v);
    bf16x8_to_f32(b, v + 8);
  }
}

template <bool kSeg>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t it = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (it >= p.num_items) return;
  if (p.live_rows != nullptr && it / p.num_heads >= static_cast<int64_t>(*p.live_rows)) return;
  const int n = p.num_parts;

  // statistic of part s: base-2 max (segments) or natural-log lse (states)
  auto stat = [&](int s) -> float {
    if constexpr (kSeg) return p.segm_max[it * n + s];
    else return p.part_lse[static_cast<int64_t>(s) * p.num_items + it];
  };
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, stat(s));
  M = warp_max(M);

  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
  uint4 *dst = reinterpret_cast<uint4 *>(p.out + it * 512 + lane * 16);
  if (M == -INFINITY) {
    dst[0] = make_uint4(0, 0, 0, 0);
    dst[1] = make_uint4(0, 0, 0, 0);
    if (lane == 0) p.lse[it] = -INFINITY;
    return;
  }

  // denominator
  float den = 0.0f;
  for (int s = lane; s < n; s += 32) {
    const float m = stat(s);
    if (m != -INFINITY) {
      if constexpr (kSeg) den += exp2f(m - M) * p.segm_sum[it * n + s];
      else den += expf(m - M);
    }
  }
  den = warp_sum(den);
  const float inv_den = 1.0f / den;

  // weighted sum, parts in chunks of 32 (lane s%32 holds part s's weight)
  for (int base = 0; base < n; base += 32) {
    float wgt = 0.0f;
    if (base + lane < n) {
      const float m = stat(base + lane);
      if (m != -INFINITY) wgt = (kSeg ? exp2f(m - M) : expf(m - M)) * inv_den;
    }
    const int cnt = min(32, n - base);
    for (int s0 = 0; s0 < cnt; s0 += 4) {
      float v[4][16];
      float w4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sl = s0 + u;
        w4[u] = __shfl_sync(0xffffffffu, wgt, sl & 31);
        if (sl < cnt && w4[u] != 0.0f) {
          load_part<kSeg>(p, it, base + sl, lane, v[u]);
        } else {
          w4[u] = 0.0f;
#pragma unroll
          for (int k = 0; k < 16; ++k) v[u][k] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = fmaf(w4[u], v[u][k], acc[k]);
    }
  }
  dst[0] = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                      pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
  dst[1] = make_uint4(pack_bf16(acc[8], acc[9]), pack_bf16(acc[10], acc[11]),
                      pack_bf16(acc[12], acc[13]), pack_bf16(acc[14], acc[15]));
  if (lane == 0) p.lse[it] = kSeg ? (M + log2f(den)) * kLn2 : M + logf(den);
}

}  // namespace

mla_status launch_merge(const MergeLaunch &m, cudaStream_t stream) {
  MergeParams p{};
  p.segm_out = m.segm_out;
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
  const int64_t blocks = (p.num_items + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (m.mode == MLA_MERGE_SEGMENTS)
    merge_kernel<true><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(p);
  else
    merge_kernel<false><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return MLA_OK;
}

}  // namespace mla
