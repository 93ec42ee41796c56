// mla_api.cu -- the C ABI of libmla_gb300.so: host-side validation, the row
// plan / shard row view integer kernels, the device error word, TMA
// descriptor encoding and the decode -> segment-merge sequence.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "mla_gb300.h"
#include "mla_internal.h"

namespace mla {

namespace {
thread_local char g_last_error[512] = "";
__device__ int g_device_error;  // first device-detected problem (mla_device_error)
// Per-device caches filled on first use.  Two host threads may fill one at
// the same time; both store the same value, so relaxed atomics suffice.
std::atomic<int *> g_err_ptr[64];
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

__device__ __forceinline__ void dev_error(int *err, int code) { atomicCAS(err, 0, code); }

// Round-robin count of window w on rank r of W (interleave 1): positions
// g < w with g mod W == r, i.e. floor((w - 1 - r) / W) + 1 when w - 1 - r >= 0.
// [vLLM #51705 digest, _build_dcp_verify_row_view snippet; sglang #34432,
// g(j) = j * W + r]
__device__ __forceinline__ int rr_count(int w, int W, int r) {
  const int top = w - 1 - r;
  return top >= 0 ? top / W + 1 : 0;
}
// Interleave I > 1 (runs of I consecutive positions dealt to the ranks in
// turn; the pages stop at I = 1): I positions per full cycle of I * W plus
// the rank's part of the last, partial cycle.
__device__ __forceinline__ int il_count(int w, int W, int r, int I) {
  if (I == 1) return rr_count(w, W, r);
  if (w <= 0) return 0;
  const int64_t cycle = static_cast<int64_t>(I) * W;
  int64_t rem = w % cycle - static_cast<int64_t>(r) * I;
  rem = rem < 0 ? 0 : (rem > I ? I : rem);
  return static_cast<int>((w / cycle) * I + rem);
}

// Request owning row r: the b with qo_indptr[b] <= r < qo_indptr[b+1].
__device__ __forceinline__ int find_request(const int32_t *ind, int B, int r) {
  int lo = 0, hi = B;  // invariant: ind[lo] <= r < ind[hi] when indptr is valid
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ind[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Sub-page row of one request [vLLM #51705 digest, 实现拆解 3]: local page p
// is block_table[b][p / R] * R + p % R (R = block_size / P) for the pages
// that hold `len` tokens, -1 after that.  Run by one block.
__device__ void subpage_row(int b, int len, const int32_t *bt, int bt_stride, int num_blocks,
                            int block_size, int P, int32_t *sp, int sp_stride, int *err) {
  int pages = (len + P - 1) / P;
  if (pages > sp_stride) {
    if (threadIdx.x == 0) dev_error(err, MLA_DEV_LEN_BOUND);
    pages = sp_stride;
  }
  const int R = block_size / P;
  int32_t *row = sp + static_cast<int64_t>(b) * sp_stride;
  for (int pg = threadIdx.x; pg < sp_stride; pg += blockDim.x) {
    int32_t v = -1;
    if (pg < pages) {
      const int bi = pg / R;
      const int blk = bi < bt_stride ? bt[static_cast<int64_t>(b) * bt_stride + bi] : -1;
      if (blk < 0 || blk >= num_blocks) dev_error(err, MLA_DEV_BAD_BLOCK_ID);
      else v = blk * R + pg % R;
    }
    row[pg] = v;
  }
}

struct TableArgs {
  const int32_t *bt;
  int bt_stride, num_blocks, block_size, P;
  int32_t *sp;
  int sp_stride;
};

// Row plan [vLLM #51705 digest, 实现拆解 2]: row t of request b sees global
// positions [0, L_b - qlen_b + t].  Blocks [0, row_blocks) write the rows;
// blocks row_blocks + b expand request b's block table (its longest row sees
// all L_b tokens) when a table is given.
__global__ void plan_kernel(int B, int T, const int32_t *seq_lens, const int32_t *ind,
                            int32_t *row_len, int32_t *row_req, TableArgs tab, int row_blocks,
                            int *err) {
  grid_dep_wait();
  grid_dep_launch();
  const int total = ind[B];
  const bool ind_ok = ind[0] == 0 && total >= 0 && total <= T;
  if (blockIdx.x >= row_blocks) {
    const int b = blockIdx.x - row_blocks;
    const int qlen = ind[b + 1] - ind[b];
    const int L = seq_lens[b];
    const int len = (ind_ok && qlen >= 1 && qlen <= L) ? L : 0;
    subpage_row(b, len, tab.bt, tab.bt_stride, tab.num_blocks, tab.block_size, tab.P, tab.sp,
                tab.sp_stride, err);
    return;
  }
  const int stride = row_blocks * blockDim.x;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += stride) {
    const int qlen = ind[b + 1] - ind[b];
    if (qlen < 0) dev_error(err, MLA_DEV_BAD_INDPTR);
    else if (qlen == 0 || qlen > seq_lens[b]) dev_error(err, MLA_DEV_BAD_QLEN);
  }
  if (!ind_ok && blockIdx.x == 0 && threadIdx.x == 0) dev_error(err, MLA_DEV_BAD_INDPTR);
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < T; r += stride) {
    if (!ind_ok || r >= total) {
      row_len[r] = 0;
      row_req[r] = -1;
      continue;
    }
    const int b = find_request(ind, B, r);
    const int qlen = ind[b + 1] - ind[b];
    const int L = seq_lens[b];
    const int t = r - ind[b];
    const bool good = qlen >= 1 && qlen <= L && t >= 0 && t < qlen;
    row_len[r] = good ? L - qlen + 1 + t : 0;
    row_req[r] = b;
  }
}

// Shard row view: per-row shard-local count from the row's global window;
// blocks row_blocks + b expand the shard's table for request b, sized by its
// longest shard-local row.  blockIdx.y selects the rank (rank0 + y) when
// several views are computed in one launch; view y's outputs and block table
// sit at the given per-view strides.
__global__ void shard_kernel(int B, int T, const int32_t *ind, const int32_t *row_len_global,
                             int W, int rank0, int I, int32_t *row_len_local, TableArgs tab,
                             int row_blocks, int *err, int64_t bt_view_stride, int64_t sp_view_stride) {
  grid_dep_wait();
  grid_dep_launch();
  const int rank = rank0 + static_cast<int>(blockIdx.y);
  row_len_local += static_cast<int64_t>(blockIdx.y) * T;
  if (tab.bt != nullptr) {
    tab.bt += static_cast<int64_t>(blockIdx.y) * bt_view_stride;
    tab.sp += static_cast<int64_t>(blockIdx.y) * sp_view_stride;
  }
  const int total = ind[B];
  const bool ind_ok = ind[0] == 0 && total >= 0 && total <= T;
  if (blockIdx.x >= row_blocks) {
    const int b = blockIdx.x - row_blocks;
    int len = 0;
    const int r0 = ind[b], r1 = ind[b + 1];
    if (ind_ok && r0 >= 0 && r1 >= r0 && r1 <= T)
      for (int r = r0; r < r1; ++r) len = max(len, il_count(row_len_global[r], W, rank, I));
    subpage_row(b, len, tab.bt, tab.bt_stride, tab.num_blocks, tab.block_size, tab.P, tab.sp,
                tab.sp_stride, err);
    return;
  }
  if (!ind_ok && blockIdx.x == 0 && threadIdx.x == 0) dev_error(err, MLA_DEV_BAD_INDPTR);
  const int stride = row_blocks * blockDim.x;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < T; r += stride) {
    row_len_local[r] = (ind_ok && r < total) ? il_count(row_len_global[r], W, rank, I) : 0;
  }
}

int grid_for(int n, int threads) {
  int g = (n + threads - 1) / threads;
  return g < 1 ? 1 : (g > 1024 ? 1024 : g);
}

bool is_aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

mla_status cuda_fail(cudaError_t e, const char *what) {
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

int *device_error_word() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return nullptr;
  }
  int *cached = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (cached == nullptr) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) {
      cuda_fail(e, "cudaGetSymbolAddress(device error word)");
      return nullptr;
    }
    cached = static_cast<int *>(ptr);
    g_err_ptr[dev].store(cached, std::memory_order_relaxed);
  }
  return cached;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  PFN_cuTensorMapEncodeTiled_v12000 fn = g_encode.load(std::memory_order_relaxed);
  if (fn != nullptr) return fn;
  void *sym = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &sym, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || sym == nullptr) {
    set_error("cuTensorMapEncodeTiled entry point unavailable");
    return nullptr;
  }
  fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(sym);
  g_encode.store(fn, std::memory_order_relaxed);
  return fn;
}

mla_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                        int elem_bytes, uint64_t cols, uint64_t rows, uint32_t box_cols,
                        uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return MLA_ERR_CUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (CUresult %d): rows=%llu cols=%llu box=%ux%u", (int)r,
              (unsigned long long)rows, (unsigned long long)cols, box_cols, box_rows);
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status make_tmap_tile3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                            int elem_bytes, uint64_t rows, uint32_t box_rows,
                            CUtensorMapSwizzle swizzle) {
  // A latent row of 576 values seen as 9 chunks of 64: dims (64 values, row,
  // chunk) with strides (row = 576 values, chunk = 64 values), so one box of
  // (64, box_rows, 9) lands chunk-major in shared memory: chunk c at
  // c * box_rows * 64 * elem_bytes, rows inside a chunk contiguous.
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return MLA_ERR_CUDA;
  const uint64_t eb = static_cast<uint64_t>(elem_bytes);
  const cuuint64_t dims[3] = {64, rows, 9};
  const cuuint64_t strides[2] = {576 * eb, 64 * eb};
  const cuuint32_t box[3] = {64, box_rows, 9};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled (3-D tile view) failed (CUresult %d): rows=%llu box_rows=%u", (int)r,
              (unsigned long long)rows, box_rows);
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status launch_plan_rows(int B, int T, const int32_t *seq_lens, const int32_t *ind,
                            int32_t *row_len, int32_t *row_req, const TableLaunch &t,
                            int *err, cudaStream_t stream) {
  const int row_blocks = grid_for(T > B ? T : B, 256);
  TableArgs tab{t.block_table, t.bt_stride, t.num_blocks, t.block_size, t.page_size,
                t.subpage_table, t.sp_stride};
  const int blocks = row_blocks + (t.block_table != nullptr ? B : 0);
  const cudaError_t e = launch_pdl(plan_kernel, dim3(blocks), dim3(256), 0, stream, B, T, seq_lens, ind, row_len,
                                   row_req, tab, row_blocks, err);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "plan_rows launch");
}

mla_status launch_shard_rows(int B, int T, const int32_t *ind, const int32_t *row_len_global,
                             int W, int rank, int num_views, int interleave, int32_t *row_len_local,
                             const TableLaunch &t, int *err, cudaStream_t stream) {
  const int row_blocks = grid_for(T, 256);
  TableArgs tab{t.block_table, t.bt_stride, t.num_blocks, t.block_size, t.page_size,
                t.subpage_table, t.sp_stride};
  const int blocks = row_blocks + (t.block_table != nullptr ? B : 0);
  const int64_t bt_view = static_cast<int64_t>(B) * t.bt_stride, sp_view = static_cast<int64_t>(B) * t.sp_stride;
  const cudaError_t e = launch_pdl(shard_kernel, dim3(blocks, num_views), dim3(256), 0, stream, B, T, ind,
                                   row_len_global, W, rank, interleave, row_len_local, tab, row_blocks, err,
                                   bt_view, sp_view);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "shard_row_view launch");
}

WorkspaceLayout decode_workspace_layout(const mla_decode_args &a) {
  WorkspaceLayout l{};
  size_t off = 0;
  if (a.num_segments > 1) {
    const size_t V = a.num_views > 1 ? a.num_views : 1;
    const size_t items = V * a.num_rows * a.num_heads * a.num_segments;
    const size_t row_blocks = (static_cast<size_t>(a.max_qlen) * a.num_heads + 63) / 64;
    const size_t blocks = V * a.num_reqs * row_blocks * a.num_segments;
    l.segm_out = off;
    off += align256(blocks * 512 * 64 * sizeof(uint16_t));
    l.segm_max = off;
    off += align256(items * sizeof(float));
    l.segm_sum = off;
    off += align256(items * sizeof(float));
  }
  l.sched = off;
  off += 256;
  l.unit_state = off;
  if (a.num_segments > 1) {
    const size_t V = a.num_views > 1 ? a.num_views : 1;
    const size_t row_blocks = (static_cast<size_t>(a.max_qlen) * a.num_heads + 63) / 64;
    off += align256(V * a.num_reqs * row_blocks * sizeof(unsigned));
  }
  l.total = off;
  return l;
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char *mla_last_error_string(void) { return g_last_error; }

const char *mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_CHECK: return "MLA_ERR_DEVICE_CHECK";
    default: return "MLA_STATUS_UNKNOWN";
  }
}

int mla_page_size(int block_size) {
  if (block_size <= 0) return -1;
  const int low_bit = block_size & -block_size;  // largest power-of-two divisor
  return low_bit < 128 ? low_bit : 128;
}

static mla_status check_table_args(const int32_t *block_table, int bt_stride, int num_blocks,
                                   int block_size, const int32_t *sp, int sp_stride, int *P_out) {
  const int P = mla_page_size(block_size);
  if (P < 0) {
    set_error("block_size must be positive (got %d)", block_size);
    return MLA_ERR_INVALID_ARG;
  }
  if (block_table != nullptr) {
    if (bt_stride < 1 || num_blocks < 1 || sp == nullptr || sp_stride < 1) {
      set_error("block table given but block_table_stride=%d num_blocks=%d subpage_stride=%d",
                bt_stride, num_blocks, sp_stride);
      return MLA_ERR_INVALID_ARG;
    }
    if (static_cast<int64_t>(num_blocks) * (block_size / P) > INT32_MAX) {
      set_error("num_blocks * (block_size / page_size) overflows int32 sub-page ids");
      return MLA_ERR_INVALID_ARG;
    }
  }
  *P_out = P;
  return MLA_OK;
}

mla_status mla_plan_rows(int num_reqs, int num_rows, const int32_t *seq_lens,
                         const int32_t *qo_indptr, int32_t *row_len, int32_t *row_req,
                         const int32_t *block_table, int block_table_stride, int num_blocks,
                         int block_size, int32_t *subpage_table, int subpage_stride,
                         mla_stream_t stream) {
  if (num_reqs < 0 || num_rows < 0 || qo_indptr == nullptr ||
      (num_reqs > 0 && seq_lens == nullptr) || (num_rows > 0 && (row_len == nullptr || row_req == nullptr))) {
    set_error("mla_plan_rows: bad sizes or null pointers (B=%d T=%d)", num_reqs, num_rows);
    return MLA_ERR_INVALID_ARG;
  }
  int P = 0;
  if (block_table != nullptr) {
    mla_status st = check_table_args(block_table, block_table_stride, num_blocks, block_size,
                                     subpage_table, subpage_stride, &P);
    if (st != MLA_OK) return st;
  }
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TableLaunch t{block_table, block_table_stride, num_blocks, block_size, P, subpage_table,
                subpage_stride};
  return launch_plan_rows(num_reqs, num_rows, seq_lens, qo_indptr, row_len, row_req, t, err, s);
}

mla_status mla_shard_row_view(int num_reqs, int num_rows, const int32_t *qo_indptr,
                              const int32_t *row_len_global, int world_size, int rank,
                              int interleave, int32_t *row_len_local, const int32_t *block_table,
                              int block_table_stride, int num_blocks, int block_size,
                              int32_t *subpage_table, int subpage_stride, mla_stream_t stream) {
  if (world_size < 1 || rank < 0 || rank >= world_size || interleave < 1 ||
      static_cast<int64_t>(interleave) * world_size > INT32_MAX) {
    set_error("mla_shard_row_view: rank %d of world_size %d, interleave %d", rank, world_size, interleave);
    return MLA_ERR_INVALID_ARG;
  }
  if (num_reqs < 0 || num_rows < 0 || qo_indptr == nullptr ||
      (num_rows > 0 && (row_len_global == nullptr || row_len_local == nullptr))) {
    set_error("mla_shard_row_view: bad sizes or null pointers (B=%d T=%d)", num_reqs, num_rows);
    return MLA_ERR_INVALID_ARG;
  }
  int P = 0;
  if (block_table != nullptr) {
    mla_status st = check_table_args(block_table, block_table_stride, num_blocks, block_size,
                                     subpage_table, subpage_stride, &P);
    if (st != MLA_OK) return st;
  }
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TableLaunch t{block_table, block_table_stride, num_blocks, block_size, P, subpage_table,
                subpage_stride};
  return launch_shard_rows(num_reqs, num_rows, qo_indptr, row_len_global, world_size, rank, 1,
                           interleave, row_len_local, t, err, s);
}

mla_status mla_shard_row_views(int num_reqs, int num_rows, const int32_t *qo_indptr,
                               const int32_t *row_len_global, int world_size, int interleave,
                               int32_t *row_len_local, const int32_t *block_tables,
                               int block_table_stride, int num_blocks, int block_size,
                               int32_t *subpage_tables, int subpage_stride, mla_stream_t stream) {
  if (world_size < 1 || world_size > 65535 || interleave < 1 ||
      static_cast<int64_t>(interleave) * world_size > INT32_MAX) {
    set_error("mla_shard_row_views: world_size %d, interleave %d", world_size, interleave);
    return MLA_ERR_INVALID_ARG;
  }
  if (num_reqs < 0 || num_rows < 0 || qo_indptr == nullptr ||
      (num_rows > 0 && (row_len_global == nullptr || row_len_local == nullptr))) {
    set_error("mla_shard_row_views: bad sizes or null pointers (B=%d T=%d)", num_reqs, num_rows);
    return MLA_ERR_INVALID_ARG;
  }
  int P = 0;
  if (block_tables != nullptr) {
    mla_status st = check_table_args(block_tables, block_table_stride, num_blocks, block_size,
                                     subpage_tables, subpage_stride, &P);
    if (st != MLA_OK) return st;
  }
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TableLaunch t{block_tables, block_table_stride, num_blocks, block_size, P, subpage_tables,
                subpage_stride};
  return launch_shard_rows(num_reqs, num_rows, qo_indptr, row_len_global, world_size, 0, world_size,
                           interleave, row_len_local, t, err, s);
}

static mla_status check_decode_args(const mla_decode_args *a) {
  if (a == nullptr) {
    set_error("mla_decode_verify: null argument struct");
    return MLA_ERR_INVALID_ARG;
  }
  if (a->num_reqs < 1 || a->num_rows < 1 || a->num_heads < 1 || a->max_qlen < 1 ||
      a->num_segments < 1 || a->subpage_stride < 1 || a->num_cache_rows < 1) {
    set_error("mla_decode_verify: B=%d T=%d H=%d max_qlen=%d S=%d subpage_stride=%d rows=%lld must be >= 1",
              a->num_reqs, a->num_rows, a->num_heads, a->max_qlen, a->num_segments,
              a->subpage_stride, (long long)a->num_cache_rows);
    return MLA_ERR_INVALID_ARG;
  }
  if (a->kv_dtype != MLA_KV_BF16 && a->kv_dtype != MLA_KV_FP8_E4M3) {
    set_error("mla_decode_verify: unknown kv_dtype %d", a->kv_dtype);
    return MLA_ERR_UNSUPPORTED;
  }
  if (a->page_size < 8 || a->page_size > 128 || (a->page_size & (a->page_size - 1)) != 0) {
    set_error("mla_decode_verify: page_size %d unsupported (power of two in [8, 128])", a->page_size);
    return MLA_ERR_UNSUPPORTED;
  }
  if (static_cast<int64_t>(a->subpage_stride) * a->page_size > INT32_MAX ||
      a->num_cache_rows > INT32_MAX || static_cast<int64_t>(a->num_rows) * a->num_heads > INT32_MAX ||
      static_cast<int64_t>(a->max_qlen) * a->num_heads > INT32_MAX) {
    set_error("mla_decode_verify: sizes overflow int32 indexing");
    return MLA_ERR_INVALID_ARG;
  }
  if (a->max_qlen > a->num_rows) {
    set_error("mla_decode_verify: max_qlen %d above the row capacity %d", a->max_qlen, a->num_rows);
    return MLA_ERR_INVALID_ARG;
  }
  if (a->wait_cycles < 0) {
    set_error("mla_decode_verify: wait_cycles must be >= 0 (0 = default)");
    return MLA_ERR_INVALID_ARG;
  }
  if (a->num_segments > kMaxParts) {
    set_error("mla_decode_verify: num_segments %d above the supported %d", a->num_segments, kMaxParts);
    return MLA_ERR_UNSUPPORTED;
  }
  if (a->q == nullptr || a->kv_cache == nullptr || a->qo_indptr == nullptr || a->row_len == nullptr ||
      a->subpage_table == nullptr || a->out == nullptr || a->lse == nullptr) {
    set_error("mla_decode_verify: null device pointer");
    return MLA_ERR_INVALID_ARG;
  }
  if (!is_aligned(a->q, 16) || !is_aligned(a->kv_cache, 16) || !is_aligned(a->out, 16)) {
    set_error("mla_decode_verify: q, kv_cache and out must be 16-byte aligned");
    return MLA_ERR_INVALID_ARG;
  }
  if (a->num_views < 0 || static_cast<int64_t>(a->num_views > 1 ? a->num_views : 1) * a->num_rows * a->num_heads > INT32_MAX ||
      static_cast<int64_t>(a->num_views > 1 ? a->num_views : 1) * a->num_reqs > INT32_MAX) {
    set_error("mla_decode_verify: num_views %d (rows x heads x views must fit int32)", a->num_views);
    return MLA_ERR_INVALID_ARG;
  }
  if ((a->flags & ~(MLA_DECODE_SKIP_MERGE | MLA_DECODE_UNIFORM_SEGMENTS | MLA_DECODE_FUSED_MERGE)) != 0) {
    set_error("mla_decode_verify: unknown flags 0x%x", a->flags);
    return MLA_ERR_INVALID_ARG;
  }
  if ((a->flags & MLA_DECODE_FUSED_MERGE) &&
      ((a->flags & (MLA_DECODE_SKIP_MERGE | MLA_DECODE_UNIFORM_SEGMENTS)) || a->num_segments < 2)) {
    set_error("mla_decode_verify: MLA_DECODE_FUSED_MERGE needs num_segments > 1 and neither "
              "MLA_DECODE_SKIP_MERGE nor MLA_DECODE_UNIFORM_SEGMENTS");
    return MLA_ERR_UNSUPPORTED;
  }
  if (!(a->sm_scale > 0.0f) || (a->kv_dtype == MLA_KV_FP8_E4M3 && !(a->kv_scale > 0.0f))) {
    set_error("mla_decode_verify: sm_scale and (fp8) kv_scale must be positive");
    return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

size_t mla_decode_verify_workspace(const mla_decode_args *a) {
  if (a == nullptr || a->num_rows < 1 || a->num_heads < 1 || a->num_segments < 1) return 0;
  return decode_workspace_layout(*a).total;
}

mla_status mla_decode_verify(const mla_decode_args *a, void *workspace, size_t workspace_bytes,
                             mla_stream_t stream) {
  mla_status st = check_decode_args(a);
  if (st != MLA_OK) return st;
  const WorkspaceLayout lay = decode_workspace_layout(*a);
  if (workspace == nullptr || workspace_bytes < lay.total || !is_aligned(workspace, 256)) {
    set_error("mla_decode_verify: workspace of %zu bytes (256-byte aligned) needed, got %zu at %p",
              lay.total, workspace_bytes, workspace);
    return MLA_ERR_WORKSPACE;
  }
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *w = static_cast<char *>(workspace);
  DecodeLaunch d{};
  d.a = a;
  d.err = err;
  d.sched = reinterpret_cast<int *>(w + lay.sched);
  d.unit_state = reinterpret_cast<unsigned *>(w + lay.unit_state);
  d.state_bytes = lay.total - lay.sched;
  const bool partials = a->num_segments > 1;
  if (partials) {
    d.segm_out = reinterpret_cast<uint16_t *>(w + lay.segm_out);
    d.segm_max = reinterpret_cast<float *>(w + lay.segm_max);
    d.segm_sum = reinterpret_cast<float *>(w + lay.segm_sum);
  }
  bool merged = false;
  st = launch_decode(d, s, &merged);
  if (st != MLA_OK || !partials || merged || (a->flags & MLA_DECODE_SKIP_MERGE)) return st;
  MergeLaunch m{};
  m.mode = MLA_MERGE_SEGMENTS;
  m.num_rows = a->num_rows;
  m.num_heads = a->num_heads;
  m.num_parts = a->num_segments;
  m.segm_out = d.segm_out;
  m.segm_max = d.segm_max;
  m.segm_sum = d.segm_sum;
  m.qo_indptr = a->qo_indptr;
  m.num_reqs = a->num_reqs;
  m.num_views = a->num_views > 1 ? a->num_views : 1;
  m.row_blocks = (a->max_qlen * a->num_heads + 63) / 64;
  m.out = a->out;
  m.lse = a->lse;
  return launch_merge(m, s);
}

mla_status mla_merge_segments(const mla_merge_args *a, mla_stream_t stream) {
  if (a == nullptr || a->num_rows < 0 || a->num_heads < 1 || a->num_parts < 1 ||
      a->out == nullptr || a->lse == nullptr) {
    set_error("mla_merge_segments: bad arguments");
    return MLA_ERR_INVALID_ARG;
  }
  if (a->num_parts > kMaxParts) {
    set_error("mla_merge_segments: num_parts %d above the supported %d", a->num_parts, kMaxParts);
    return MLA_ERR_UNSUPPORTED;
  }
  if (a->mode == MLA_MERGE_SEGMENTS) {
    if (a->segm_out == nullptr || a->segm_max == nullptr || a->segm_sum == nullptr ||
        a->qo_indptr == nullptr || !is_aligned(a->segm_out, 16)) {
      set_error("mla_merge_segments: segment mode needs 16-byte aligned segm_out, segm_max, segm_sum and qo_indptr");
      return MLA_ERR_INVALID_ARG;
    }
    if (a->num_reqs < 0 || a->max_qlen < 1 || a->num_views < 0 ||
        static_cast<int64_t>(a->max_qlen) * a->num_heads > INT32_MAX ||
        static_cast<int64_t>(a->num_views > 1 ? a->num_views : 1) * a->num_rows * a->num_heads > INT32_MAX) {
      set_error("mla_merge_segments: bad num_reqs %d / max_qlen %d / num_views %d", a->num_reqs, a->max_qlen,
                a->num_views);
      return MLA_ERR_INVALID_ARG;
    }
  } else if (a->mode == MLA_MERGE_STATES) {
    if (a->part_out == nullptr || a->part_lse == nullptr || !is_aligned(a->part_out, 16)) {
      set_error("mla_merge_segments: state mode needs 16-byte aligned part_out and part_lse");
      return MLA_ERR_INVALID_ARG;
    }
  } else {
    set_error("mla_merge_segments: unknown mode %d", a->mode);
    return MLA_ERR_INVALID_ARG;
  }
  if (!is_aligned(a->out, 16)) {
    set_error("mla_merge_segments: out must be 16-byte aligned");
    return MLA_ERR_INVALID_ARG;
  }
  MergeLaunch m{};
  m.mode = a->mode;
  m.num_rows = a->num_rows;
  m.num_heads = a->num_heads;
  m.num_parts = a->num_parts;
  m.segm_out = a->segm_out;
  m.segm_max = a->segm_max;
  m.segm_sum = a->segm_sum;
  m.qo_indptr = a->qo_indptr;
  m.num_reqs = a->num_reqs;
  m.num_views = a->num_views > 1 ? a->num_views : 1;
  m.row_blocks = a->mode == MLA_MERGE_SEGMENTS ? (a->max_qlen * a->num_heads + 63) / 64 : 0;
  m.part_out = a->part_out;
  m.part_lse = a->part_lse;
  m.out = a->out;
  m.lse = a->lse;
  return launch_merge(m, reinterpret_cast<cudaStream_t>(stream));
}

mla_status mla_get_device_error(int32_t *code_out, mla_stream_t stream) {
  if (code_out == nullptr) {
    set_error("mla_get_device_error: null code_out");
    return MLA_ERR_INVALID_ARG;
  }
  *code_out = 0;
  int *err = device_error_word();
  if (err == nullptr) return MLA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int code = 0;
  cudaError_t e = cudaMemcpyAsync(&code, err, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_get_device_error");
  *code_out = code;
  return code == 0 ? MLA_OK : MLA_ERR_DEVICE_CHECK;
}

}  // extern "C"
