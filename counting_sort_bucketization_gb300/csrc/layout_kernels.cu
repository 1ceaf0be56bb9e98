// layout_kernels.cu -- count, column scan and stable rank of the MoE
// dispatch layout (counting sort / bucketization) on sm_103a.
//
// Method: page "07 DeepEP Counting Sort / Bucketization", [CS] below.
//   count   [CS] §4.2: per-expert counts and per-rank counts with one count
//           per token per rank.  As on the page, each CTA first counts in a
//           shared-memory histogram and warps deduplicate ranks with
//           __match_any_sync; unlike the page, the per-CTA histograms are
//           kept (one column per tile) instead of being reduced into one
//           global array, because the stable scatter needs every tile's base.
//   scan    [CS] §5.2-§5.5, §7.2: the page scans on one SM after a grid-wide
//           reduction; here one warp per expert scans that expert's tile
//           column, and every rank CTA recomputes the (small) aligned
//           exclusive sum over experts itself, so no kernel waits on another
//           SM inside a launch.
//   rank    [CS] §6.4 assigns slots with atomicAdd on the exclusive sum,
//           which makes the order inside a segment depend on scheduling.
//           Here the slot is expert_offset[e] + (pairs of e in earlier
//           tiles) + (pairs of e earlier in this tile), the last term from
//           __match_any_sync + popc within a warp and a per-expert scan over
//           the warps: token-ascending and deterministic.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Stage the tile's topk ids into shared memory as int32: masked -> -1,
// id >= E -> -1 and flagged.
__device__ __forceinline__ void stage_tile_ids(const int64_t* __restrict__ topk_idx,
                                               int64_t pair0, int npairs, int E, int* ids_s,
                                               int* err) {
  bool bad = false;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    const int64_t v = __ldg(topk_idx + pair0 + i);
    int e = -1;
    if (v >= 0) {
      if (v < E)
        e = static_cast<int>(v);
      else
        bad = true;
    }
    ids_s[i] = e;
  }
  if (bad) set_error(err, MOE_ERR_BAD_EXPERT_ID);
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < kWarpSize; d <<= 1) {
    const int u = __shfl_up_sync(kFull, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

// ----------------------------------------------------------------- count
__global__ void __launch_bounds__(kLayoutThreads)
    count_tiles_kernel(const int64_t* __restrict__ topk_idx, int64_t N, int K, int E, int R,
                       TilePlan plan, int32_t* __restrict__ hist, int32_t* __restrict__ rhist,
                       int* err) {
  extern __shared__ int smem[];
  int* hist_s = smem;         // [E]
  int* rhist_s = smem + E;    // [R]
  int* ids_s = rhist_s + R;   // [tile pairs]
  const int tile = blockIdx.x;
  const int64_t T = plan.tiles;
  const int64_t t0 = static_cast<int64_t>(tile) * plan.tile_tokens;
  const int ntok = static_cast<int>(min64(plan.tile_tokens, N - t0));
  const int L = E / R;

  for (int i = threadIdx.x; i < E + R; i += blockDim.x) smem[i] = 0;
  stage_tile_ids(topk_idx, t0 * K, ntok * K, E, ids_s, err);
  __syncthreads();

  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int tok_in_chunk = lane / K;
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < ntok;
    const int e = in ? ids_s[chunk * plan.lanes + lane] : -1;
    const bool valid = e >= 0;
    // Experts: one shared atomic per distinct expert in the chunk.
    const unsigned peers = __match_any_sync(kFull, valid ? static_cast<unsigned>(e)
                                                         : (0x80000000u | lane));
    if (valid && __ffs(peers) - 1 == lane) atomicAdd(&hist_s[e], __popc(peers));
    // Ranks: lanes of the same token that hit the same rank form one group;
    // only its lowest lane counts ([CS] §4.2 deduplication).
    const int r = valid ? e / L : 0;
    const unsigned rkey = valid ? static_cast<unsigned>(tok_in_chunk * MOE_MAX_EXPERTS + r)
                                : (0x80000000u | lane);
    const unsigned rpeers = __match_any_sync(kFull, rkey);
    if (valid && __ffs(rpeers) - 1 == lane) atomicAdd(&rhist_s[r], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(e) * T + tile] = hist_s[e];
  for (int r = threadIdx.x; r < R; r += blockDim.x) rhist[static_cast<int64_t>(r) * T + tile] = rhist_s[r];
}

// ----------------------------------------------------------- column scan
// One warp per row: expert rows become exclusive prefixes over tiles and
// give expert_count; rank rows give rank_count.
__global__ void __launch_bounds__(kLayoutThreads)
    scan_columns_kernel(int32_t* __restrict__ hist, const int32_t* __restrict__ rhist, int64_t T,
                        int E, int R, int32_t* __restrict__ expert_count,
                        int32_t* __restrict__ rank_count) {
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int row = blockIdx.x * kLayoutWarps + warp;
  if (row >= E + R) return;
  const bool is_expert = row < E;
  const int32_t* src = is_expert ? hist + static_cast<int64_t>(row) * T
                                 : rhist + static_cast<int64_t>(row - E) * T;
  const int64_t m = ceil_div64(T, kWarpSize);
  const int64_t lo = min64(lane * m, T), hi = min64(lo + m, T);
  int sum = 0;
  for (int64_t i = lo; i < hi; ++i) sum += src[i];
  const int incl = warp_inclusive_scan(sum, lane);
  const int total = __shfl_sync(kFull, incl, kWarpSize - 1);
  if (is_expert) {
    int32_t* dst = hist + static_cast<int64_t>(row) * T;
    int run = incl - sum;
    for (int64_t i = lo; i < hi; ++i) {
      const int c = dst[i];
      dst[i] = run;
      run += c;
    }
    if (lane == 0) expert_count[row] = total;
  } else if (lane == 0) {
    rank_count[row - E] = total;
  }
}

// ------------------------------------------------------------ rank + maps
__global__ void __launch_bounds__(kLayoutThreads)
    rank_maps_kernel(const int64_t* __restrict__ topk_idx, int64_t N, int K, int E, int R, int A,
                     TilePlan plan, const int32_t* __restrict__ hist_prefix,
                     const int32_t* __restrict__ expert_count,
                     const int32_t* __restrict__ rank_count, int32_t* __restrict__ expert_offset,
                     int32_t* __restrict__ rank_psum, int32_t* __restrict__ dst_slot,
                     int32_t* __restrict__ src_idx, int64_t capacity, int32_t* __restrict__ total_rows,
                     int* err) {
  extern __shared__ int smem[];
  int* off_s = smem;                          // [E+1] aligned exclusive offsets
  int* cnt_s = off_s + (E + 1);               // [kLayoutWarps][E] per-warp counters, then bases
  int* ids_s = cnt_s + kLayoutWarps * E;      // [tile pairs]
  int* lr_s = ids_s + plan.tile_tokens * K;   // [tile pairs] rank inside the warp's run
  __shared__ int warp_tot_s[kLayoutWarps];

  const int tile = blockIdx.x;
  const int64_t T = plan.tiles;
  const int64_t t0 = static_cast<int64_t>(tile) * plan.tile_tokens;
  const int ntok = static_cast<int>(max64(0, min64(plan.tile_tokens, N - t0)));
  const int npairs = ntok * K;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;

  for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) cnt_s[i] = 0;
  stage_tile_ids(topk_idx, t0 * K, npairs, E, ids_s, err);

  // Aligned exclusive sum over experts ([CS] §7.2 then §5.5), block-wide.
  // Thread i owns experts [i*ipt, (i+1)*ipt).
  const int ipt = static_cast<int>(ceil_div64(E, kLayoutThreads));
  const int e_lo = threadIdx.x * ipt;
  int mine = 0;
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) mine += static_cast<int>(ceil_div64(__ldg(expert_count + e), A) * A);
  }
  const int incl = warp_inclusive_scan(mine, lane);
  if (lane == kWarpSize - 1) warp_tot_s[warp] = incl;
  __syncthreads();
  int warp_base = 0;
  for (int w = 0; w < warp; ++w) warp_base += warp_tot_s[w];
  int run = warp_base + incl - mine;
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) {
      off_s[e] = run;
      run += static_cast<int>(ceil_div64(__ldg(expert_count + e), A) * A);
    }
  }
  if (threadIdx.x == kLayoutThreads - 1) off_s[E] = run;
  __syncthreads();
  const int64_t rows = off_s[E];
  const bool cap_ok = rows <= capacity;

  if (tile == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offset[e] = off_s[e];
    if (threadIdx.x == 0) {
      *total_rows = static_cast<int32_t>(rows);
      if (!cap_ok) set_error(err, MOE_ERR_CAPACITY);
    }
    if (warp == 0) {  // inclusive sum over ranks ([CS] §5.5)
      int carry = 0;
      for (int base = 0; base < R; base += kWarpSize) {
        const int r = base + lane;
        const int v = r < R ? __ldg(rank_count + r) : 0;
        const int s = warp_inclusive_scan(v, lane) + carry;
        if (r < R) rank_psum[r] = s;
        carry = __shfl_sync(kFull, s, kWarpSize - 1);
      }
    }
  }

  // Rank of each pair among the same expert's pairs earlier in its warp's run.
  const int tok_in_chunk = lane / K;
  int* my_cnt = cnt_s + warp * E;
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < ntok;
    const int pair = chunk * plan.lanes + lane;
    const int e = in ? ids_s[pair] : -1;
    const bool valid = e >= 0;
    const unsigned peers = __match_any_sync(kFull, valid ? static_cast<unsigned>(e)
                                                         : (0x80000000u | lane));
    const int base = valid ? my_cnt[e] : 0;
    __syncwarp();
    if (valid) {
      if (__ffs(peers) - 1 == lane) my_cnt[e] = base + __popc(peers);
      lr_s[pair] = base + __popc(peers & ptx::lanemask_lt());
    }
    __syncwarp();
  }
  __syncthreads();

  // Per expert: turn the per-warp counts into absolute slot bases.
  for (int e = threadIdx.x; e < E && tile < T; e += blockDim.x) {
    int b = off_s[e] + hist_prefix[static_cast<int64_t>(e) * T + tile];
    for (int w = 0; w < kLayoutWarps; ++w) {
      const int c = cnt_s[w * E + e];
      cnt_s[w * E + e] = b;
      b += c;
    }
  }
  __syncthreads();

  // Maps, in flat (t, k) order (coalesced dst_slot writes).
  const int pairs_per_warp = plan.cpw * plan.lanes;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    const int e = ids_s[i];
    int slot = -1;
    if (e >= 0 && cap_ok) {
      slot = cnt_s[(i / pairs_per_warp) * E + e] + lr_s[i];
      src_idx[slot] = static_cast<int32_t>(t0 + i / K);
    }
    dst_slot[t0 * K + i] = slot;
  }

  // Alignment-gap rows have no source token.
  if (cap_ok) {
    for (int e = tile; e < E; e += gridDim.x) {
      const int lo = off_s[e] + __ldg(expert_count + e), hi = off_s[e + 1];
      for (int row = lo + threadIdx.x; row < hi; row += blockDim.x) src_idx[row] = -1;
    }
  }
}

}  // namespace

size_t count_smem_bytes(const moe_layout_desc& d, const TilePlan& p) {
  return sizeof(int) * (static_cast<size_t>(d.num_experts) + d.num_ranks +
                        static_cast<size_t>(p.tile_tokens) * d.topk);
}

size_t rank_smem_bytes(const moe_layout_desc& d, const TilePlan& p) {
  return sizeof(int) * (static_cast<size_t>(d.num_experts) + 1 +
                        static_cast<size_t>(kLayoutWarps) * d.num_experts +
                        2 * static_cast<size_t>(p.tile_tokens) * d.topk);
}

cudaError_t launch_count(const moe_layout_desc& d, const TilePlan& p, const int64_t* topk_idx,
                         int32_t* expert_count, int32_t* rank_count, int* err, int32_t* hist,
                         int32_t* rhist, cudaStream_t stream) {
  const size_t smem1 = count_smem_bytes(d, p);
  cudaError_t st = cudaFuncSetAttribute(count_tiles_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem1));
  if (st != cudaSuccess) return st;
  if (p.tiles > 0) {
    count_tiles_kernel<<<static_cast<unsigned>(p.tiles), kLayoutThreads, smem1, stream>>>(
        topk_idx, d.num_tokens, d.topk, d.num_experts, d.num_ranks, p, hist, rhist, err);
    count_launch();
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
  }
  const int rows = d.num_experts + d.num_ranks;
  scan_columns_kernel<<<(rows + kLayoutWarps - 1) / kLayoutWarps, kLayoutThreads, 0, stream>>>(
      hist, rhist, p.tiles, d.num_experts, d.num_ranks, expert_count, rank_count);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_rank(const moe_layout_desc& d, const TilePlan& p, const int64_t* topk_idx,
                        const int32_t* hist_prefix, const int32_t* expert_count,
                        const int32_t* rank_count, int32_t* expert_offset, int32_t* rank_psum,
                        int32_t* dst_slot, int32_t* src_idx, int64_t capacity,
                        int32_t* total_rows, int* err, cudaStream_t stream) {
  const size_t smem = rank_smem_bytes(d, p);
  cudaError_t st = cudaFuncSetAttribute(rank_maps_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
  if (st != cudaSuccess) return st;
  const int64_t grid = p.tiles > 0 ? p.tiles : 1;
  rank_maps_kernel<<<static_cast<unsigned>(grid), kLayoutThreads, smem, stream>>>(
      topk_idx, d.num_tokens, d.topk, d.num_experts, d.num_ranks, d.alignment, p, hist_prefix,
      expert_count, rank_count, expert_offset, rank_psum, dst_slot, src_idx, capacity,
      total_rows, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace moe
