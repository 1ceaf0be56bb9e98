// moe_layout_noalloc.cu -- moe_layout_build_noalloc(): the one-call layout
// (count, prefix sums, slot maps) for callers that cannot allocate device
// memory, with its scratch in a fixed array that is part of this library.
//
// Some callers cannot call cudaMalloc at the point where they build the
// layout: a serving engine that reserves all of HBM for its own allocator
// at start-up and forbids allocations afterwards, a plugin that must not
// touch the host application's memory pool, or a latency-critical loop where
// cudaMalloc's implicit device-wide synchronisation is not acceptable.  They
// still own their inputs and outputs; only the scratch (the workspace of the
// other entry points) comes from here.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {
namespace {

// The scratch.  Every GPU that loads the library holds these
// MOE_NOALLOC_SCRATCH_BYTES until the process exits; all calls on a device
// share it.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
std::vector<void*> g_scratch_addr;   // per device; nullptr until that device is set up

// Device address of the scratch on the current device.  The first call on a
// device looks it up (cudaGetSymbolAddress, with that device current) and
// caches it; later calls only read the cache.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (dev >= static_cast<int>(g_scratch_addr.size())) g_scratch_addr.resize(dev + 1, nullptr);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_layout_build_noalloc(const moe_layout_desc* desc, const int64_t* topk_idx,
                                        int32_t* expert_count, int32_t* rank_count, int32_t* expert_offset,
                                        int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx,
                                        int64_t capacity_rows, int32_t* total_rows, int32_t* device_error,
                                        void* stream) {
  size_t need = 0;
  if (int st = moe_layout_workspace_bytes(desc, &need)) return st;
  if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;   // problem too big for the fixed scratch
  if (device_error == nullptr) return MOE_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (int st = moe::scratch_address(&scratch)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The error word and the grid-barrier words must start at zero; the
  // histograms are rewritten in full by every call.
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (int st = moe_layout_build(desc, topk_idx, expert_count, rank_count, scratch, need, expert_offset, rank_psum,
                                dst_slot, src_idx, capacity_rows, total_rows, stream))
    return st;
  // This call's device-side status: the scratch's error word.
  if (cudaMemcpyAsync(device_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
