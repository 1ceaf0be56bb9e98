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
#include "launch.h"

namespace moe {
namespace {

// The scratch.  Every GPU that loads the library holds these
// MOE_NOALLOC_SCRATCH_BYTES until the process exits; all calls on a device
// share it.
__device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch in each CUDA context seen so far.
struct ScratchAddr {
  uint64_t ctx;   // current_context_id() of the context
  void* ptr;
};
std::mutex g_scratch_mu;
std::vector<ScratchAddr> g_scratch_addr;

// Device address of the scratch in the current context.  The first call in a
// context (the first on a device, and again the first after a device reset
// has replaced that device's context) looks it up with cudaGetSymbolAddress,
// with that device current, and caches it; later calls only read the cache.
int scratch_address(void** out) {
  const uint64_t ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (const ScratchAddr& a : g_scratch_addr)
      if (a.ctx == ctx) {
        *out = a.ptr;
        return MOE_OK;
      }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_status(e);
  if (p == nullptr) return cuda_status(cudaErrorInvalidSymbol);
  // With no context current before the lookup (ctx == 0) the lookup made one;
  // the next call caches its address.
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    g_scratch_addr.push_back(ScratchAddr{ctx, p});
  }
  *out = p;
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
  if (cudaError_t e = cudaMemsetAsync(scratch, 0, 256, s)) return moe::cuda_status(e);
  if (int st = moe_layout_build(desc, topk_idx, expert_count, rank_count, scratch, need, expert_offset, rank_psum,
                                dst_slot, src_idx, capacity_rows, total_rows, stream))
    return st;
  // This call's device-side status: the scratch's error word.
  if (cudaError_t e = cudaMemcpyAsync(device_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s))
    return moe::cuda_status(e);
  return MOE_OK;
}
