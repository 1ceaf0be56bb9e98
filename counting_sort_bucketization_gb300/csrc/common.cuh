// common.cuh -- definitions shared by the library's kernels and its C-ABI
// host code: the tile plan of the count / rank kernels, the workspace layout,
// the sticky device error word and the kernel-launch counter.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "moe_layout.h"  // include/ is on the include path

namespace moe {

constexpr int kWarpSize = 32;
constexpr int kLayoutWarps = 8;                        // warps per count / rank CTA
constexpr int kLayoutThreads = kLayoutWarps * kWarpSize;
constexpr int kMaxChunksPerWarp = 16;
#ifndef MOE_LAYOUT_TARGET_TILES
#define MOE_LAYOUT_TARGET_TILES 256
#endif
constexpr int kTargetTiles = MOE_LAYOUT_TARGET_TILES;   // tiles the plan aims for
constexpr uint64_t kWaitLimitNs = 1000000000ull;       // 1 s bound on any in-kernel wait

// The count and rank kernels walk topk_idx in token-aligned chunks of one warp:
// a chunk holds tpc = 32 / K whole tokens (tpc * K <= 32 lanes busy), a warp
// walks cpw consecutive chunks and a CTA (tile) holds kLayoutWarps warps.
// Pairs (t, k) of a tile are contiguous in topk_idx, so a tile's pairs in
// (warp, chunk, lane) order are exactly its pairs in (t, k) order.
struct TilePlan {
  int tpc;           // tokens per chunk
  int lanes;         // busy lanes per chunk = tpc * K
  int cpw;           // chunks per warp
  int tile_tokens;   // tokens per tile = kLayoutWarps * cpw * tpc
  int64_t tiles;     // T = ceil(N / tile_tokens)
};

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

inline TilePlan make_tile_plan(int64_t N, int K) {
  TilePlan p;
  p.tpc = kWarpSize / K;
  p.lanes = p.tpc * K;
  const int64_t per_cpw = static_cast<int64_t>(kLayoutWarps) * p.tpc;
  int64_t cpw = ceil_div64(N, per_cpw * kTargetTiles);
  if (cpw < 1) cpw = 1;
  if (cpw > kMaxChunksPerWarp) cpw = kMaxChunksPerWarp;
  p.cpw = static_cast<int>(cpw);
  p.tile_tokens = static_cast<int>(per_cpw * cpw);
  p.tiles = ceil_div64(N, p.tile_tokens);
  return p;
}

// Workspace: [error word, grid-barrier words | pad to 256 B][hist int32 E x T]
// [rank hist int32 R x T].  hist[e][tile] is expert e's count in the tile;
// the column scan turns it into the count of expert e in all earlier tiles.
struct WorkspaceLayout {
  size_t err_off = 0;
  size_t bar_off = 16;   // two unsigned: grid-barrier arrival counter (zero between launches), spare
  size_t work_off = 32;  // four unsigned: permute's unit counter, its finished CTAs; the combine's two
  size_t hist_off = 256;
  size_t rhist_off = 0;
  size_t bytes = 0;
};

inline WorkspaceLayout make_workspace_layout(const moe_layout_desc& d, const TilePlan& p) {
  WorkspaceLayout w;
  const size_t T = static_cast<size_t>(p.tiles);
  w.rhist_off = w.hist_off + ((static_cast<size_t>(d.num_experts) * T * 4 + 255) / 256) * 256;
  w.bytes = w.rhist_off + ((static_cast<size_t>(d.num_ranks) * T * 4 + 255) / 256) * 256;
  return w;
}

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel on the stream is still running; it must execute
// griddepcontrol.wait (ptx::grid_dependency_wait) before it reads anything
// that kernel may write.  With any other predecessor (a copy, a kernel that
// never triggers) it behaves like an ordinary launch.
//
// Every kernel of this library triggers its dependents only after its own
// griddepcontrol.wait has returned.  So when a kernel of the library starts,
// everything before its immediate predecessor on the stream has completed,
// and it may read before its wait whatever no kernel of the library writes:
// the routing ids (topk_idx) and the token rows and scale rows (x, sf).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// An ordinary launch (no attributes) through cudaLaunchKernelEx.
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// Counter behind moe_kernel_launches().
void count_launch(int n = 1);

// MOE_OK for cudaSuccess; otherwise records `e` as this thread's last CUDA
// error (moe_last_cuda_error) and returns MOE_ERR_CUDA.  Every MOE_ERR_CUDA
// the library returns goes through it.
int cuda_status(cudaError_t e);

}  // namespace moe
