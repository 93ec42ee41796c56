// mla_noalloc.cu -- mla_decode_verify for callers that cannot allocate device
// memory.
//
// mla_decode_verify needs a scratch workspace (split-K partials and a work
// counter) that the caller allocates.  Some callers cannot do that at the
// point of the call: serving runtimes that reserve all device memory at
// start-up and forbid allocation on the request path; plugin hosts and plain
// C callers that hold no device allocator and for which a cudaMalloc would
// synchronise the device in the middle of a step.  This file gives them one
// more entry point whose scratch is a fixed-size array in the library's own
// device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "mla_gb300.h"
#include "mla_internal.h"

namespace mla {
namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(MLA_STATIC_SCRATCH_BYTES);
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the array, per device (relaxed atomic: two threads making
// their first call at once store the same value).
std::atomic<void *> g_static_scratch_ptr[64];

// The array's name is a host-side stand-in in host code: its device address
// is looked up once per device, with that device current.
mla_status static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return MLA_ERR_CUDA;
  }
  void *ptr = g_static_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (ptr == nullptr) {
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_scratch_ptr[dev].store(ptr, std::memory_order_relaxed);
  }
  *out = ptr;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_decode_verify_noalloc(const mla_decode_args *a, mla_stream_t stream) {
  if (a == nullptr) {
    mla::set_error("mla_decode_verify_noalloc: null argument struct");
    return MLA_ERR_INVALID_ARG;
  }
  const size_t need = mla_decode_verify_workspace(a);
  if (need > mla::kStaticScratchBytes) {
    mla::set_error(
        "mla_decode_verify_noalloc: this problem needs %zu bytes of scratch (rows x heads x "
        "segments too large); the library's static scratch holds %zu bytes -- use "
        "mla_decode_verify with a workspace",
        need, mla::kStaticScratchBytes);
    return MLA_ERR_WORKSPACE;
  }
  void *scratch = nullptr;
  const mla_status st = mla::static_scratch(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode_verify(a, scratch, mla::kStaticScratchBytes, stream);
}
