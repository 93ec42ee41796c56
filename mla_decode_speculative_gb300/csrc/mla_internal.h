// mla_internal.h -- declarations shared by the translation units of
// libmla_gb300.so (host launchers, error plumbing).  Not part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_gb300.h"

namespace mla {

// Records a printf-style message as the calling thread's last error text.
void set_error(const char *fmt, ...);
// Records a CUDA runtime failure and returns MLA_ERR_CUDA.
mla_status cuda_fail(cudaError_t e, const char *what);

// Device address of the library's device error word on the current device
// (looked up once per device); nullptr after recording an error.
int *device_error_word();

// Encodes a 2-D tiled TMA descriptor over a row-major [rows, cols] matrix.
mla_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                        int elem_bytes, uint64_t cols, uint64_t rows, uint32_t box_cols,
                        uint32_t box_rows, CUtensorMapSwizzle swizzle);
// 3-D view of a [rows, 576] latent cache for whole-tile boxes (64 values x
// box_rows x 9 chunks, chunk-major in shared memory).
mla_status make_tmap_tile3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                            int elem_bytes, uint64_t rows, uint32_t box_rows,
                            CUtensorMapSwizzle swizzle);

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization: its CTAs may be scheduled while the
// kernel before it in the stream is still finishing, run their prologue
// (barriers, tensor memory), and then block in grid_dep_wait() until that
// kernel has completed and its memory is visible -- before their first
// global-memory access, read or write.  grid_dep_launch() lets the next
// kernel's CTAs be scheduled (they still wait for this grid to complete).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Launchers (arguments already validated on the host).
struct TableLaunch {  // optional sub-page expansion (block_table == nullptr: none)
  const int32_t *block_table;
  int bt_stride, num_blocks, block_size, page_size;
  int32_t *subpage_table;
  int sp_stride;
};
mla_status launch_plan_rows(int num_reqs, int num_rows, const int32_t *seq_lens,
                            const int32_t *qo_indptr, int32_t *row_len, int32_t *row_req,
                            const TableLaunch &table, int *err, cudaStream_t stream);
// Views rank .. rank + num_views - 1 (blockIdx.y), outputs and tables at
// per-view strides T, B * sp_stride and B * bt_stride.
mla_status launch_shard_rows(int num_reqs, int num_rows, const int32_t *qo_indptr,
                             const int32_t *row_len_global, int world_size, int rank, int num_views,
                             int interleave, int32_t *row_len_local, const TableLaunch &table,
                             int *err, cudaStream_t stream);

struct DecodeLaunch {
  const mla_decode_args *a;
  uint16_t *segm_out;  // bf16
  float *segm_max;
  float *segm_sum;
  int *sched;           // work-claim counter (workspace), zeroed before a launch that reads it
  unsigned *unit_state; // per-unit part counters (workspace, after sched), zeroed with it
  size_t state_bytes;   // bytes from sched through the unit counters
  int *err;
};
// Workspace layout of mla_decode_verify: [segm_out][segm_max][segm_sum] (only
// when num_segments > 1, 256-byte aligned regions), then 256 bytes of work
// counter, then (num_segments > 1) one 32-bit counter per (view, request,
// 64-row block) unit.
struct WorkspaceLayout {
  size_t segm_out, segm_max, segm_sum, sched, unit_state, total;
};
WorkspaceLayout decode_workspace_layout(const mla_decode_args &a);
// Launches the decode.  *merged is set when the kernel also merged the
// split-K parts into out / lse itself (balanced split), so no merge launch
// must follow.
mla_status launch_decode(const DecodeLaunch &d, cudaStream_t stream, bool *merged);

struct MergeLaunch {
  int mode;
  int num_rows;
  int num_heads;
  int num_parts;
  const uint16_t *segm_out;  // bf16 blocks [B, RB, S, 8, 512, 8]
  const float *segm_max;
  const float *segm_sum;
  const int32_t *qo_indptr;  // segment mode
  int num_reqs;              // segment mode
  int num_views;             // segment mode: V row views (>= 1)
  int row_blocks;            // segment mode: RB
  const void *part_out;
  const float *part_lse;
  void *out;
  float *lse;
};
mla_status launch_merge(const MergeLaunch &m, cudaStream_t stream);

constexpr int kMaxParts = 1024;  // most split-K segments / shards one merge combines

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace mla
