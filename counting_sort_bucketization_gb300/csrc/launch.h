// launch.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace moe {

size_t count_smem_bytes(const moe_layout_desc& d, const TilePlan& p);
size_t rank_smem_bytes(const moe_layout_desc& d, const TilePlan& p);

// topk_idx as int64 (the default) or int32.
struct IdsRef {
  const void* ptr;
  bool i32;
};

// count_tiles_kernel + scan_columns_kernel.
cudaError_t launch_count(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, int32_t* expert_count,
                         int32_t* rank_count, int* err, int32_t* hist, int32_t* rhist, cudaStream_t stream);

// rank_maps_kernel.
cudaError_t launch_rank(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, const int32_t* hist_prefix,
                        const int32_t* expert_count, const int32_t* rank_count, int32_t* expert_offset,
                        int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx, int64_t capacity,
                        int32_t* total_rows, int* err, cudaStream_t stream);

// Count + scan + rank: one cooperative kernel when every tile fits on the
// GPU at once, else the three kernels above.
cudaError_t launch_build(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, int32_t* expert_count,
                         int32_t* rank_count, int32_t* hist, int32_t* rhist, unsigned* barrier_words,
                         int32_t* expert_offset, int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx,
                         int64_t capacity, int32_t* total_rows, int* err, cudaStream_t stream);

// cumulative[e] += expert_count[e] (int64 running totals across calls).
cudaError_t launch_accumulate_stats(const int32_t* expert_count, int E, int64_t* cumulative, cudaStream_t stream);

// rank_rows_kernel: the non-expand (rank-contiguous) slot map.
cudaError_t launch_rank_rows(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, const int32_t* rhist_prefix,
                             const int32_t* rank_count, int32_t* rank_slot, int32_t* rank_src, int64_t capacity,
                             int* err, cudaStream_t stream);

struct PermuteArgs {
  const uint8_t* x;
  const uint8_t* sf;
  int64_t row_bytes;
  int64_t sf_row_bytes;
  const int32_t* dst_slot;
  const int32_t* total_rows;     // rows the layout uses (checked against capacity)
  const int32_t* expert_offset;  // gap rows (zero_pad only)
  const int32_t* expert_count;
  uint8_t* recv_x;
  uint8_t* recv_sf;
  int64_t capacity;
  int64_t num_tokens;
  int topk;
  int num_experts;
  int zero_pad;
  int* err;
  unsigned* work;                // [2] token counter + finished-CTA counter (zero between launches)
  bool non_expand;               // rows of the non-expand layout (sizes the dynamic kernel's pieces)
  uint64_t wait_ns;              // bound on each mbarrier wait (set by launch_permute)
  unsigned extra_tx;             // test hook: bytes no copy delivers, on each CTA's first stage
};

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t stream);

struct CombineArgs {
  const uint16_t* expert_out;  // bf16 bits
  int64_t expert_out_rows;
  int64_t hidden;
  const int32_t* dst_slot;
  const float* weights;
  uint16_t* out;               // bf16 bits
  int64_t num_tokens;
  int topk;
  int* err;
  unsigned* work;              // [2] token counter + finished-CTA counter (zero between launches)
  uint64_t wait_ns;            // bound on each mbarrier wait (set by launch_combine)
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

struct SfColMajorArgs {
  const uint32_t* sf;          // [num_tokens, cols] 4-byte scale words
  int64_t cols;
  const int32_t* src;          // token of each receive row; -1 = gap row
  const int32_t* total_rows;   // rows in use (checked against capacity)
  uint32_t* out;               // column j at out + j * ld
  int64_t ld;
  int64_t capacity;
  int64_t num_tokens;
  int zero_pad;
  int* err;
};

cudaError_t launch_sf_col_major(const SfColMajorArgs& a, cudaStream_t stream);

// Limit of every in-kernel wait and the test hooks that make a wait run out
// (moe_debug_set_waits); the launchers copy them into the kernels' arguments.
struct WaitConfig {
  uint64_t limit_ns;        // bound on any in-kernel wait (default kWaitLimitNs)
  unsigned barrier_extra;   // added to the fused layout's grid-barrier targets (0 in normal use)
  unsigned extra_tx;        // bytes added to each CTA's first permute stage (0 in normal use)
};
WaitConfig wait_config();

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Host-side launch settings, looked up once instead of on every call.
//   ensure_smem_limit: raise `func`'s dynamic shared-memory limit to at least
//     `smem` bytes in the current context; the runtime call is made only when
//     the limit must grow (cached per context, so a context created after a
//     device reset sets it again).
//   cached_occupancy: resident CTAs per SM of `func` at (threads, smem) on
//     the current device, 0 if the query failed (then not cached).
//   cooperative_launch_supported: the current device's attribute, cached.
//   current_context_id: a nonzero identity of the current context, 0 if none.
cudaError_t ensure_smem_limit(const void* func, size_t smem);
int cached_occupancy(const void* func, int threads, size_t smem);
bool cooperative_launch_supported();
uint64_t current_context_id();

template <typename... KArgs>
cudaError_t ensure_smem_limit(void (*func)(KArgs...), size_t smem) {
  return ensure_smem_limit(reinterpret_cast<const void*>(func), smem);
}
template <typename... KArgs>
int cached_occupancy(void (*func)(KArgs...), int threads, size_t smem) {
  return cached_occupancy(reinterpret_cast<const void*>(func), threads, smem);
}

}  // namespace moe
