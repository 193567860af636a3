// sinkattn_decode_static_scratch: decode whose split scratch is a fixed
// device array inside the library, for callers that cannot allocate device
// memory.  It hands that array to the shared decode entry as the workspace,
// asking it to clear the merge counters once every check has passed.

#include "sinkattn.h"
#include "kernels.cuh"

#include <cuda_runtime.h>

#include <atomic>

namespace {

constexpr int kMaxDevices = 64;

// The scratch itself: one copy per device that loads the library, kept until
// the process exits.
__device__ __align__(256) unsigned char g_decode_scratch[SINKATTN_STATIC_SCRATCH_BYTES];

// Device address of g_decode_scratch per device.  In host code the symbol
// name is only a host-side handle, never a device pointer.
std::atomic<void *> g_scratch_ptr[kMaxDevices];

int scratch_for_current_device(void **ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SINKATTN_CUDA_ERROR;
  }
  void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SINKATTN_CUDA_ERROR;
    }
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  return SINKATTN_OK;
}

}  // namespace

extern "C" SINKATTN_API int sinkattn_decode_static_scratch(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *page_table,
    int max_pages_per_seq, const int32_t *kv_lens, const float *sinks, float scale, void *out,
    float *lse, int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
    int num_pages, int max_kv_len, int num_splits, void *stream) {
  void *scratch = nullptr;
  if (batch > 0) {
    const int st = scratch_for_current_device(&scratch);
    if (st != SINKATTN_OK) return st;
  }
  // decode_entry runs every argument check and the plan first; only a plan
  // with more than one split then clears its merge counters (the first bytes
  // of the array, within the plan's workspace size, which the size check
  // keeps within the array) before the launch.  A refused call queues
  // nothing, and a single-split call touches nothing in the array.
  return sa::decode_entry(q, k_cache, v_cache, page_table, max_pages_per_seq, kv_lens, nullptr,
                         sinks, scale, out, lse, batch, 1, num_qo_heads, num_kv_heads, head_dim,
                         page_size, num_pages, max_kv_len, num_splits, scratch,
                         SINKATTN_STATIC_SCRATCH_BYTES, SINKATTN_LAUNCH_DEFAULT, true, stream);
}
