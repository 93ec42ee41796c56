// mla_kvwrite.cu -- owner-filtered write of the new verify tokens into a
// (context-sharded) paged latent KV cache.
//
// sglang #34432 digest, 实现拆解 4 (set_mla_kv_buffer filters by owner and
// divides by the shard count) and key snippet g(j) = j * W + r: request b's
// qlen_b new tokens sit at global positions g = L_b - qlen_b + t; rank r of W
// keeps those with g mod W == r, at its local index j = g div W, i.e. cache row
// block_table[b][j / block_size] * block_size + j % block_size.  bf16 caches
// receive the 576 values unchanged; fp8 caches receive the e4m3 codes of
// (value / kv_scale) in float32, rounded to nearest even and saturated.
//
// Memory-bound scatter: one warp per new token row, 16-byte loads and stores.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

struct WriteParams {
  const int32_t *seq_lens;
  const int32_t *qo_indptr;
  const uint4 *kv_new;  // [T, 576] bf16 as 72 x 16-byte chunks per row
  const int32_t *block_table;
  void *cache;
  int *err;
  int64_t cache_rows;
  int num_reqs, num_rows, world_size, rank, interleave, bt_stride, num_blocks, block_size;
  float kv_scale;
  int fp8;
};

__device__ __forceinline__ int owner_request(const int32_t *ind, int B, int r) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ind[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

__global__ void write_kv_kernel(const WriteParams p) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int total = p.qo_indptr[p.num_reqs];
  if (p.qo_indptr[0] != 0 || total < 0 || total > p.num_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(p.err, 0, MLA_DEV_BAD_INDPTR);
    return;
  }
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < total; r += warps) {
    const int b = owner_request(p.qo_indptr, p.num_reqs, r);
    const int qlen = p.qo_indptr[b + 1] - p.qo_indptr[b];
    const int L = p.seq_lens[b];
    if (qlen < 1 || qlen > L) {
      if (lane == 0) atomicCAS(p.err, 0, MLA_DEV_BAD_QLEN);
      continue;
    }
    const int g = L - qlen + (r - p.qo_indptr[b]);
    // owner: runs of I positions dealt to the ranks in turn (I = 1: g mod W)
    if ((g / p.interleave) % p.world_size != p.rank) continue;  // another shard owns this token
    const int j = static_cast<int>((g / (static_cast<int64_t>(p.interleave) * p.world_size)) * p.interleave +
                                   g % p.interleave);
    const int bi = j / p.block_size;
    const int blk = bi < p.bt_stride ? p.block_table[static_cast<int64_t>(b) * p.bt_stride + bi] : -1;
    const int64_t slot = static_cast<int64_t>(blk) * p.block_size + j % p.block_size;
    if (blk < 0 || blk >= p.num_blocks || slot >= p.cache_rows) {
      if (lane == 0) atomicCAS(p.err, 0, MLA_DEV_BAD_BLOCK_ID);
      continue;
    }
    const uint4 *src = p.kv_new + static_cast<int64_t>(r) * 72;
    if (!p.fp8) {
      uint4 *dst = static_cast<uint4 *>(p.cache) + slot * 72;
      for (int i = lane; i < 72; i += 32) dst[i] = src[i];
    } else {
      uint2 *dst = static_cast<uint2 *>(p.cache) + slot * 72;
      for (int i = lane; i < 72; i += 32) {
        const uint4 u = src[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t out[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float a0 = __uint_as_float(w[2 * k] << 16) / p.kv_scale;
          const float a1 = __uint_as_float(w[2 * k] & 0xffff0000u) / p.kv_scale;
          const float a2 = __uint_as_float(w[2 * k + 1] << 16) / p.kv_scale;
          const float a3 = __uint_as_float(w[2 * k + 1] & 0xffff0000u) / p.kv_scale;
          const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
          const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a2, a3), __NV_SATFINITE, __NV_E4M3);
          out[k] = lo | (hi << 16);
        }
        dst[i] = make_uint2(out[0], out[1]);
      }
    }
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_write_kv(int num_reqs, int num_rows, const int32_t *seq_lens,
                                   const int32_t *qo_indptr, const void *kv_new, int world_size,
                                   int rank, int interleave, const int32_t *block_table,
                                   int block_table_stride, int num_blocks, int block_size,
                                   void *kv_cache, int kv_dtype, float kv_scale,
                                   int64_t num_cache_rows, mla_stream_t stream) {
  if (num_reqs < 0 || num_rows < 0 || world_size < 1 || rank < 0 || rank >= world_size ||
      interleave < 1 || static_cast<int64_t>(interleave) * world_size > INT32_MAX ||
      block_size < 1 || block_table_stride < 1 || num_blocks < 1 || num_cache_rows < 1 ||
      (num_reqs > 0 && (seq_lens == nullptr || qo_indptr == nullptr || block_table == nullptr)) ||
      (num_rows > 0 && kv_new == nullptr) || kv_cache == nullptr) {
    set_error("mla_write_kv: bad sizes or null pointers (B=%d T=%d W=%d rank=%d block=%d)", num_reqs,
              num_rows, world_size, rank, block_size);
    return MLA_ERR_INVALID_ARG;
  }
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) {
    set_error("mla_write_kv: unknown kv_dtype %d", kv_dtype);
    return MLA_ERR_UNSUPPORTED;
  }
  if (kv_dtype == MLA_KV_FP8_E4M3 && !(kv_scale > 0.0f)) {
    set_error("mla_write_kv: fp8 kv_scale must be positive");
    return MLA_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(kv_new) | reinterpret_cast<uintptr_t>(kv_cache)) % 16 != 0) {
    set_error("mla_write_kv: kv_new and kv_cache must be 16-byte aligned");
    return MLA_ERR_INVALID_ARG;
  }
  if (num_reqs == 0 || num_rows == 0) return MLA_OK;
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  WriteParams p{};
  p.seq_lens = seq_lens;
  p.qo_indptr = qo_indptr;
  p.kv_new = static_cast<const uint4 *>(kv_new);
  p.block_table = block_table;
  p.cache = kv_cache;
  p.err = err;
  p.cache_rows = num_cache_rows;
  p.num_reqs = num_reqs;
  p.num_rows = num_rows;
  p.world_size = world_size;
  p.rank = rank;
  p.interleave = interleave;
  p.bt_stride = block_table_stride;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.kv_scale = kv_scale;
  p.fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const int warps_per_block = 8;
  int blocks = (num_rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 4096) blocks = 4096;
  write_kv_kernel<<<blocks, warps_per_block * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "write_kv launch");
}
