// layout_kernels.cu -- count, column scan and stable rank of the MoE
// dispatch layout (counting sort / bucketization) on sm_103a.
//
// Method: page "07 DeepEP Counting Sort / Bucketization", [CS] below.
//   count   [CS] §4.2: per-expert counts and per-rank counts with one count
//           per token per rank.  As on the page, each CTA first counts in a
//           shared-memory histogram; the rank deduplication the page does
//           with a warp match is done here from the token's own ids in shared
//           memory (a token counts in a rank on its first pair there).  Unlike
//           the page, the per-CTA histograms are kept (one column per tile)
//           instead of being reduced into one global array, because the
//           stable scatter needs every tile's base.
//   scan    [CS] §5.2-§5.5, §7.2: the page scans on one SM after a grid-wide
//           reduction; here one warp per expert scans that expert's tile
//           column, and every rank CTA recomputes the (small) aligned
//           exclusive sum over experts itself.
//   rank    [CS] §6.4 assigns slots with atomicAdd on the exclusive sum,
//           which makes the order inside a segment depend on scheduling.
//           Here the slot is expert_offset[e] + (pairs of e in earlier
//           tiles) + (pairs of e earlier in this tile), the last term from a
//           per-warp running count per expert, advanced one token at a time
//           (a token's pairs name distinct experts), and a per-expert scan
//           over the warps: token-ascending and deterministic.
//
// Two ways to run the three phases:
//   - three kernels (count_tiles, scan_columns, rank_maps), chained with
//     programmatic dependent launch: the two-call API, and the one-call build
//     until a tile holds the most chunks per warp (batches up to ~1 M pairs at
//     top-8) or when the tiles do not all fit on the GPU at once.  The rank
//     kernel stages and ranks its ids before its wait, overlapping the count
//     and the column scan;
//   - one cooperative kernel (layout_fused_kernel) with two grid barriers,
//     the one-call build at the largest tile plan when every tile's CTA fits
//     on the GPU at once.  The tile's ids stay in shared memory from the count
//     to the rank phase, and two launches and their gaps disappear.  Its
//     barrier waits are bounded (MOE_ERR_TIMEOUT).
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Stage the tile's topk ids into shared memory as int32: masked -> -1,
// id >= E -> -1 and flagged.
// Each thread issues kStageBatch independent loads before it uses any, so a
// tile of thousands of pairs costs a few memory latencies, not one per pair.
#ifndef MOE_LAYOUT_STAGE_BATCH
#define MOE_LAYOUT_STAGE_BATCH 8
#endif
constexpr int kStageBatch = MOE_LAYOUT_STAGE_BATCH;

template <typename IdT>
__device__ __forceinline__ void stage_tile_ids(const IdT* __restrict__ topk_idx,
                                               int64_t pair0, int npairs, int E, int* ids_s,
                                               int* err) {
  bool bad = false;
  for (int base = threadIdx.x; base < npairs; base += kStageBatch * blockDim.x) {
    int64_t v[kStageBatch];
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
      const int i = base + u * blockDim.x;
      v[u] = i < npairs ? __ldg(topk_idx + pair0 + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
      const int i = base + u * blockDim.x;
      if (i >= npairs) break;
      int e = -1;
      if (v[u] >= 0) {
        if (v[u] < E)
          e = static_cast<int>(v[u]);
        else
          bad = true;
      }
      ids_s[i] = e;
    }
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

// Exclusive prefix of `mine` over the block's threads in thread order, for
// blocks whose threads each own a contiguous run of the items being summed:
// a warp scan, then the warps' totals through shared memory.  Contains a
// __syncthreads, so it also publishes the block's earlier shared writes.
__device__ __forceinline__ int block_exclusive_base(int mine, int* warp_tot_s) {
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int incl = warp_inclusive_scan(mine, lane);
  if (lane == kWarpSize - 1) warp_tot_s[warp] = incl;
  __syncthreads();
  int base = incl - mine;
  for (int w = 0; w < warp; ++w) base += warp_tot_s[w];
  return base;
}

struct TileCoords {
  int64_t t0;   // first token of the tile
  int ntok;     // tokens in the tile (the last tile may be short)
};

__device__ __forceinline__ TileCoords tile_coords(const TilePlan& plan, int64_t N, int tile) {
  TileCoords c;
  c.t0 = static_cast<int64_t>(tile) * plan.tile_tokens;
  c.ntok = static_cast<int>(max64(0, min64(plan.tile_tokens, N - c.t0)));
  return c;
}

// What pair (t, k) with expert e learns from token t's own ids (contiguous
// in the staged tile, `tok` points at the first): how many of the token's
// earlier and later pairs name e too (duplicates: the method's precondition
// excludes them, the pair-by-pair definition still orders them by k), and
// whether an earlier or a later pair of the token reaches e's rank (the
// token's last pair reaching a rank carries the non-expand row).
struct TokenView {
  int dup_before, dup_after;
  bool first_in_rank, last_in_rank;
};

__device__ __forceinline__ TokenView token_view(const int* tok, int K, int k, int e, int L) {
  TokenView v{0, 0, true, true};
  const int r_lo = (e / L) * L;
  for (int j = 0; j < K; ++j) {
    const int f = tok[j];
    if (j == k || f < 0) continue;
    if (f == e) {
      if (j < k) ++v.dup_before; else ++v.dup_after;
    }
    if (f >= r_lo && f < r_lo + L) {
      if (j < k) v.first_in_rank = false; else v.last_in_rank = false;
    }
  }
  return v;
}

// Whether this pair is the one that counts its token in rank r ([CS] §4.2:
// a token counts once in each rank it reaches).  Warp-collective: every lane
// calls it, `valid` false for lanes without a pair.  Up to 32 ranks, each
// token of the chunk gets a word of rank bits in shared memory and the pair
// whose atomicOr sets the bit counts; beyond that, a warp match on
// (token, rank).  Measured on GB300 (one-call layout of 131072 x 8 ids): the
// bit words took the rank pass from 15.4 to 10.7 us.
__device__ __forceinline__ bool counts_token_in_rank(bool valid, int tic, int r, int tpc, int R) {
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  if (R <= kWarpSize) {
    __shared__ unsigned tok_ranks_s[kLayoutWarps][kWarpSize];
    unsigned* words = tok_ranks_s[warp];
    if (lane < tpc) words[lane] = 0u;
    __syncwarp();
    bool first = false;
    if (valid) first = (atomicOr(&words[tic], 1u << r) & (1u << r)) == 0u;
    __syncwarp();
    return first;
  }
  const unsigned key = valid ? static_cast<unsigned>(tic * MOE_MAX_EXPERTS + r) : (0x80000000u | lane);
  const unsigned peers = __match_any_sync(kFull, key);
  return valid && __ffs(peers) - 1 == lane;
}

// ------------------------------------------------------- phase: count
// ids_s holds the tile's staged ids; hist_s [E] and rhist_s [R] are zeroed.
// Writes the tile's column of hist [E][T] and rhist [R][T].
__device__ void count_phase(const TilePlan& plan, int K, int E, int R, int tile, int ntok,
                            const int* ids_s, int* hist_s, int* rhist_s, int32_t* __restrict__ hist,
                            int32_t* __restrict__ rhist) {
  const int L = E / R;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int tok_in_chunk = lane / K;
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < ntok;
    const int e = in ? ids_s[chunk * plan.lanes + lane] : -1;
    const bool valid = e >= 0;
    const int r = valid ? e / L : 0;
    if (valid) atomicAdd(&hist_s[e], 1);
    if (counts_token_in_rank(valid, tok_in_chunk, r, plan.tpc, R)) atomicAdd(&rhist_s[r], 1);
  }
  __syncthreads();
  const int64_t T = plan.tiles;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(e) * T + tile] = hist_s[e];
  for (int r = threadIdx.x; r < R; r += blockDim.x) rhist[static_cast<int64_t>(r) * T + tile] = rhist_s[r];
}

// ------------------------------------------------- phase: column scan
// Warp w of CTA b scans rows b*kLayoutWarps + w, + gridDim.x*kLayoutWarps, ...
// Every row becomes an exclusive prefix over tiles (in place); expert rows
// give expert_count, rank rows rank_count.  Loads go through L2 (__ldcg): in the fused
// kernel other CTAs wrote these rows earlier in the same launch.
constexpr int kScanBatch = 8;   // 32-tile chunks of a row loaded before they are scanned

__device__ void scan_phase(int32_t* __restrict__ hist, int32_t* __restrict__ rhist, int64_t T, int E,
                           int R, int32_t* __restrict__ expert_count, int32_t* __restrict__ rank_count) {
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  for (int row = blockIdx.x * kLayoutWarps + warp; row < E + R; row += gridDim.x * kLayoutWarps) {
    const bool is_expert = row < E;
    int32_t* col = is_expert ? hist + static_cast<int64_t>(row) * T : rhist + static_cast<int64_t>(row - E) * T;
    // kScanBatch coalesced loads (32 tiles each) in flight, then one warp scan
    // per 32-tile chunk with a running carry; the row becomes an exclusive
    // prefix in place.
    int carry = 0;
    for (int64_t base = 0; base < T; base += kScanBatch * kWarpSize) {
      int v[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        const int64_t i = base + j * kWarpSize + lane;
        v[j] = i < T ? __ldcg(col + i) : 0;
      }
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        if (base + j * kWarpSize >= T) break;
        const int incl = warp_inclusive_scan(v[j], lane);
        const int64_t i = base + j * kWarpSize + lane;
        if (i < T) col[i] = carry + incl - v[j];
        carry += __shfl_sync(kFull, incl, kWarpSize - 1);
      }
    }
    if (lane == 0) {
      if (is_expert)
        expert_count[row] = carry;
      else
        rank_count[row - E] = carry;
    }
  }
}

// -------------------------------------------------- phase: rank + maps
struct RankArgs {
  int64_t N;
  int K, E, R, A;
  const int32_t* hist_prefix;   // [E][T] exclusive prefixes over tiles
  const int32_t* expert_count;
  const int32_t* rank_count;
  int32_t* expert_offset;
  int32_t* rank_psum;
  int32_t* dst_slot;
  int32_t* src_idx;
  int64_t capacity;
  int32_t* total_rows;
  int* err;
  uint64_t wait_ns;         // bound on each grid-barrier wait
  unsigned barrier_extra;   // added to the grid-barrier targets: 0 except under the timeout test hook
};

// Rank of each pair among the same expert's pairs earlier in its warp's run
// (lr_s), each warp's per-expert counts (cnt_s[warp][e], zeroed before) and
// the tile's per-expert counts (ecount_s, zeroed before).  When rhist_s is
// given, also the tile's rank counts, once per token and rank ([CS] §4.2
// deduplication): the fused kernel needs no separate count pass.
//
// The chunk's tokens are ranked one at a time: a token's pairs name distinct
// experts, so each reads its expert's running count and writes it back one
// higher, and pairs end up ranked in (t, k) order.  Measured on GB300 this
// beat a warp match per chunk (one-call layout of 131072 x 8 ids: rank pass
// 15.4 -> 10.7 us with the rank bits of counts_token_in_rank).  A token that
// names one expert twice (outside the method's precondition, but still
// defined pair by pair) would lose a count; the per-warp sums are checked
// against the tile's exact counts, and a tile that fails is ranked again with
// warp matches, which order repeated pairs by k.
__device__ void rank_pass(const TilePlan& plan, int K, int E, int R, int ntok, const int* ids_s, int* cnt_s,
                          int* lr_s, int* ecount_s, int* rhist_s) {
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int L = E / R;
  const int tok_in_chunk = lane / K;
  int* my_cnt = cnt_s + warp * E;
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < ntok;
    const int pair = chunk * plan.lanes + lane;
    const int e = in ? ids_s[pair] : -1;
    const bool valid = e >= 0;
    for (int i = 0; i < plan.tpc; ++i) {
      const bool mine = valid && tok_in_chunk == i;
      const int base = mine ? my_cnt[e] : 0;
      __syncwarp();
      if (mine) {
        my_cnt[e] = base + 1;
        lr_s[pair] = base;
      }
      __syncwarp();
    }
    if (valid) atomicAdd(&ecount_s[e], 1);
    if (rhist_s != nullptr) {
      const int r = valid ? e / L : 0;
      if (counts_token_in_rank(valid, tok_in_chunk, r, plan.tpc, R)) atomicAdd(&rhist_s[r], 1);
    }
  }
  __syncthreads();
  bool lost = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int sum = 0;
    for (int w = 0; w < kLayoutWarps; ++w) sum += cnt_s[w * E + e];
    lost |= sum != ecount_s[e];
  }
  if (!__syncthreads_or(lost)) return;
  // A repeated expert inside a token: rank the tile again, repeats in k order.
  for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) cnt_s[i] = 0;
  __syncthreads();
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < ntok;
    const int pair = chunk * plan.lanes + lane;
    const int e = in ? ids_s[pair] : -1;
    const bool valid = e >= 0;
    const unsigned peers = __match_any_sync(kFull, valid ? static_cast<unsigned>(e) : (0x80000000u | lane));
    const int base = valid ? my_cnt[e] : 0;
    __syncwarp();
    if (valid) {
      if (__ffs(peers) - 1 == lane) my_cnt[e] = base + __popc(peers);
      lr_s[pair] = base + __popc(peers & ptx::lanemask_lt());
    }
    __syncwarp();
  }
  __syncthreads();
}

// ids_s holds the tile's staged ids; cnt_s [kLayoutWarps*E] and lr_s come
// from rank_pass; off_s [E+1] and gap_s [E] are shared scratch.  Offsets,
// the tile-0 outputs, absolute slots, the maps and the gap rows of src_idx.
__device__ void rank_finish(const TilePlan& plan, const RankArgs& a, int tile, TileCoords tc, const int* ids_s,
                           int* off_s, int* gap_s, int* cnt_s, int* lr_s, int* warp_tot_s) {
  const int K = a.K, E = a.E, R = a.R, A = a.A;
  const int64_t T = plan.tiles;
  const int npairs = tc.ntok * K;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;

  // Both global reads of this phase are issued up front, so their latencies
  // overlap: the aligned counts of this thread's experts [i*ipt, (i+1)*ipt)
  // and this tile's earlier-tile counts for experts tid, tid+256, ...
  // (E <= MOE_MAX_EXPERTS = 4 * kLayoutThreads).
  constexpr int kPerThread = MOE_MAX_EXPERTS / kLayoutThreads;
  const int ipt = static_cast<int>(ceil_div64(E, kLayoutThreads));
  const int e_lo = threadIdx.x * ipt;
  int raw[kPerThread], prior[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int e = e_lo + j;
    raw[j] = (j < ipt && e < E) ? __ldcg(a.expert_count + e) : 0;
    const int e2 = threadIdx.x + j * kLayoutThreads;
    prior[j] = (e2 < E && tile < T) ? __ldcg(a.hist_prefix + static_cast<int64_t>(e2) * T + tile) : 0;
  }

  // Aligned exclusive sum over experts ([CS] §7.2 then §5.5), block-wide.
  int aligned[kPerThread];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    aligned[j] = static_cast<int>(ceil_div64(raw[j], A) * A);
    mine += aligned[j];
  }
  int run = block_exclusive_base(mine, warp_tot_s);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int e = e_lo + j;
    if (j < ipt && e < E) {
      off_s[e] = run;
      gap_s[e] = run + raw[j];   // first alignment-gap row of e
      run += aligned[j];
    }
  }
  if (threadIdx.x == kLayoutThreads - 1) off_s[E] = run;
  __syncthreads();
  const int64_t rows = off_s[E];
  const bool cap_ok = rows <= a.capacity;

  if (tile == 0) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) a.expert_offset[e] = off_s[e];
    if (threadIdx.x == 0) {
      *a.total_rows = static_cast<int32_t>(rows);
      if (!cap_ok) set_error(a.err, MOE_ERR_CAPACITY);
    }
    if (warp == 0) {  // inclusive sum over ranks ([CS] §5.5)
      int carry = 0;
      for (int base = 0; base < R; base += kWarpSize) {
        const int r = base + lane;
        const int v = r < R ? __ldcg(a.rank_count + r) : 0;
        const int s = warp_inclusive_scan(v, lane) + carry;
        if (r < R) a.rank_psum[r] = s;
        carry = __shfl_sync(kFull, s, kWarpSize - 1);
      }
    }
  }

  // Per expert: turn the per-warp counts into absolute slot bases.
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int e = threadIdx.x + j * kLayoutThreads;
    if (e < E && tile < T) {
      int b = off_s[e] + prior[j];
      for (int w = 0; w < kLayoutWarps; ++w) {
        const int c = cnt_s[w * E + e];
        cnt_s[w * E + e] = b;
        b += c;
      }
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
      a.src_idx[slot] = static_cast<int32_t>(tc.t0 + i / K);
    }
    a.dst_slot[tc.t0 * K + i] = slot;
  }

  // Alignment-gap rows have no source token: one warp per expert, the gap's
  // bounds already in shared memory (no global read per expert).
  if (cap_ok) {
    for (int e = tile * kLayoutWarps + warp; e < E; e += gridDim.x * kLayoutWarps) {
      const int hi = off_s[e + 1];
      for (int row = gap_s[e] + lane; row < hi; row += kWarpSize) a.src_idx[row] = -1;
    }
  }
}

// ---------------------------------------------------------- kernels
template <typename IdT>
__global__ void __launch_bounds__(kLayoutThreads)
    count_tiles_kernel(const IdT* __restrict__ topk_idx, int64_t N, int K, int E, int R,
                       TilePlan plan, int32_t* __restrict__ hist, int32_t* __restrict__ rhist,
                       int* err) {
  extern __shared__ int smem[];
  int* hist_s = smem;         // [E]
  int* rhist_s = smem + E;    // [R]
  int* ids_s = rhist_s + R;   // [tile pairs]
  const TileCoords tc = tile_coords(plan, N, blockIdx.x);
  for (int i = threadIdx.x; i < E + R; i += blockDim.x) smem[i] = 0;
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  stage_tile_ids(topk_idx, tc.t0 * K, tc.ntok * K, E, ids_s, err);
  __syncthreads();
  count_phase(plan, K, E, R, blockIdx.x, tc.ntok, ids_s, hist_s, rhist_s, hist, rhist);
}

__global__ void __launch_bounds__(kLayoutThreads)
    scan_columns_kernel(int32_t* __restrict__ hist, int32_t* __restrict__ rhist, int64_t T,
                        int E, int R, int32_t* __restrict__ expert_count,
                        int32_t* __restrict__ rank_count) {
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  scan_phase(hist, rhist, T, E, R, expert_count, rank_count);
}

// The rank kernels stage their tile's ids and rank them inside each warp
// before griddepcontrol.wait: the ids come from no kernel of this library, so
// that part runs while the kernel before them (the column scan, or the layout)
// is still working, and only the reads of the counts wait for it.
template <typename IdT>
__global__ void __launch_bounds__(kLayoutThreads)
    rank_maps_kernel(const IdT* __restrict__ topk_idx, TilePlan plan, RankArgs a) {
  extern __shared__ int smem[];
  int* off_s = smem;                            // [E+1]
  int* gap_s = off_s + (a.E + 1);               // [E]
  int* cnt_s = gap_s + a.E;                     // [kLayoutWarps][E]
  int* ids_s = cnt_s + kLayoutWarps * a.E;      // [tile pairs]
  int* lr_s = ids_s + plan.tile_tokens * a.K;   // [tile pairs]
  int* ecount_s = lr_s + plan.tile_tokens * a.K;   // [E]
  __shared__ int warp_tot_s[kLayoutWarps];
  const TileCoords tc = tile_coords(plan, a.N, blockIdx.x);
  for (int i = threadIdx.x; i < kLayoutWarps * a.E; i += blockDim.x) cnt_s[i] = 0;
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) ecount_s[i] = 0;
  stage_tile_ids(topk_idx, tc.t0 * a.K, tc.ntok * a.K, a.E, ids_s, a.err);
  __syncthreads();   // staged ids and zeroed counters visible to every warp
  rank_pass(plan, a.K, a.E, a.R, tc.ntok, ids_s, cnt_s, lr_s, ecount_s, nullptr);
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  rank_finish(plan, a, blockIdx.x, tc, ids_s, off_s, gap_s, cnt_s, lr_s, warp_tot_s);
}

// Grid-wide barrier for a cooperative launch on a counter that only grows
// within the launch: barrier b (1, 2, ...) is passed once the counter holds
// b * gridDim.x arrivals, so a barrier costs one atomic and the polls.  Each
// CTA arrives once more when it leaves (grid_exit); the last of those
// arrivals resets the counter for the next launch on the workspace.  The
// wait is bounded; on timeout the error word gets MOE_ERR_TIMEOUT and the CTA
// stops (the counter then stays set: the workspace must be zeroed again).
__device__ bool grid_barrier(unsigned* count, unsigned target, int* err, int* flag_s, uint64_t wait_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    __threadfence();   // the CTA's writes before the barrier, then the arrival
    atomicAdd(count, 1u);
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::ld_acquire_gpu(count) < target) {
      if (ptx::globaltimer_ns() - t0 > wait_ns) {
        set_error(err, MOE_ERR_TIMEOUT);
        ok = false;
        break;
      }
    }
    __threadfence();
    *flag_s = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag_s != 0;
}

// Last arrival: every CTA has passed all `barriers` barriers; reset the counter.
__device__ void grid_exit(unsigned* count, unsigned barriers) {
  if (threadIdx.x == 0 && atomicAdd(count, 1u) == (barriers + 1) * gridDim.x - 1) atomicExch(count, 0u);
}

template <typename IdT>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_fused_kernel(const IdT* __restrict__ topk_idx, TilePlan plan, RankArgs a, int32_t* hist,
                        int32_t* rhist, int32_t* expert_count, int32_t* rank_count, unsigned* bar) {
  extern __shared__ int smem[];
  const int E = a.E, R = a.R, K = a.K;
  int* ids_s = smem;                            // [tile pairs], kept across all phases
  int* lr_s = ids_s + plan.tile_tokens * K;     // [tile pairs]
  int* cnt_s = lr_s + plan.tile_tokens * K;     // [kLayoutWarps][E]
  int* off_s = cnt_s + kLayoutWarps * E;        // [E+1]
  int* gap_s = off_s + (E + 1);                 // [E]
  int* rhist_s = gap_s + E;                     // [R]
  int* ecount_s = rhist_s + R;                  // [E]
  __shared__ int warp_tot_s[kLayoutWarps];
  __shared__ int flag_s;
  const int tile = blockIdx.x;
  const int64_t T = plan.tiles;
  const TileCoords tc = tile_coords(plan, a.N, tile);
  for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) cnt_s[i] = 0;
  for (int i = threadIdx.x; i < R; i += blockDim.x) rhist_s[i] = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) ecount_s[i] = 0;
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  stage_tile_ids(topk_idx, tc.t0 * K, tc.ntok * K, E, ids_s, a.err);
  __syncthreads();
  // One pass over the tile's pairs: ranks inside each warp's run, per-warp
  // and per-tile expert counts, deduplicated rank counts.
  rank_pass(plan, K, E, R, tc.ntok, ids_s, cnt_s, lr_s, ecount_s, rhist_s);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(e) * T + tile] = ecount_s[e];
  for (int r = threadIdx.x; r < R; r += blockDim.x) rhist[static_cast<int64_t>(r) * T + tile] = rhist_s[r];
  if (!grid_barrier(bar, gridDim.x + a.barrier_extra, a.err, &flag_s, a.wait_ns)) return;
  scan_phase(hist, rhist, plan.tiles, E, R, expert_count, rank_count);
  if (!grid_barrier(bar, 2 * gridDim.x + a.barrier_extra, a.err, &flag_s, a.wait_ns)) return;
  grid_exit(bar, 2);
  rank_finish(plan, a, tile, tc, ids_s, off_s, gap_s, cnt_s, lr_s, warp_tot_s);
}

// ------------------------------------------- non-expand rank rows
// [CS] §6.2 (Scatter 1): one row per (token, rank) the token reaches, in
// rank r's block [start_r, start_r + rank_count[r]) where start_r is the
// exclusive sum of rank_count; tokens ascending inside a block.  The row goes
// to the token's highest k reaching r (the master lane of that token and
// rank); the other slots get -1.  The slot is start_r + (rows of r in earlier
// tiles, from the scanned rank histogram) + (rows of r earlier in this tile:
// a per-warp running count per rank advanced one token at a time, and a scan
// over the warps).
struct RankRowsArgs {
  int64_t N;
  int K, E, R;
  const int32_t* rhist_prefix;   // [R][T] exclusive prefixes over tiles
  const int32_t* rank_count;
  int32_t* rank_slot;
  int32_t* rank_src;
  int64_t capacity;
  int* err;
};

template <typename IdT>
__global__ void __launch_bounds__(kLayoutThreads)
    rank_rows_kernel(const IdT* __restrict__ topk_idx, TilePlan plan, RankRowsArgs a) {
  extern __shared__ int smem[];
  const int K = a.K, E = a.E, R = a.R, L = E / R;
  int* start_s = smem;                          // [R+1] block starts, then the total
  int* cnt_s = start_s + (R + 1);               // [kLayoutWarps][R]
  int* ids_s = cnt_s + kLayoutWarps * R;        // [tile pairs]
  int* lr_s = ids_s + plan.tile_tokens * K;     // [tile pairs] rank among masters, -1 otherwise
  __shared__ int warp_tot_s[kLayoutWarps];
  const int tile = blockIdx.x;
  const TileCoords tc = tile_coords(plan, a.N, tile);
  const int64_t T = plan.tiles;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  for (int i = threadIdx.x; i < kLayoutWarps * R; i += blockDim.x) cnt_s[i] = 0;
  // Before the wait (the ids come from no kernel of this library): stage the
  // tile and rank each token's master lanes inside its warp.
  stage_tile_ids(topk_idx, tc.t0 * K, tc.ntok * K, E, ids_s, a.err);
  __syncthreads();
  const int tok_in_chunk = lane / K, k = lane % K;
  int* my_cnt = cnt_s + warp * R;
  for (int c = 0; c < plan.cpw; ++c) {
    const int chunk = warp * plan.cpw + c;
    const int tok = chunk * plan.tpc + tok_in_chunk;
    const bool in = lane < plan.lanes && tok < tc.ntok;
    const int pair = chunk * plan.lanes + lane;
    const int e = in ? ids_s[pair] : -1;
    const bool valid = e >= 0;
    const int r = valid ? e / L : 0;
    // The master is the token's last pair reaching r.
    const bool master = valid && token_view(ids_s + pair - k, K, k, e, L).last_in_rank;
    // Masters ranked per rank in token order, the chunk's tokens one at a
    // time (a token's masters reach distinct ranks).
    for (int i = 0; i < plan.tpc; ++i) {
      const bool mine = master && tok_in_chunk == i;
      const int base = mine ? my_cnt[r] : 0;
      __syncwarp();
      if (mine) {
        my_cnt[r] = base + 1;
        lr_s[pair] = base;
      }
      __syncwarp();
    }
    if (in && !master) lr_s[pair] = -1;
  }
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();

  // Block starts: exclusive sum of rank_count (thread i owns ranks [i*ipt, (i+1)*ipt)).
  constexpr int kPerThread = MOE_MAX_EXPERTS / kLayoutThreads;
  const int ipt = static_cast<int>(ceil_div64(R, kLayoutThreads));
  const int r_lo = threadIdx.x * ipt;
  int cnt[kPerThread], prior[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int r = r_lo + j;
    cnt[j] = (j < ipt && r < R) ? __ldcg(a.rank_count + r) : 0;
    const int r2 = threadIdx.x + j * kLayoutThreads;
    prior[j] = (r2 < R && tile < T) ? __ldcg(a.rhist_prefix + static_cast<int64_t>(r2) * T + tile) : 0;
  }
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) mine += cnt[j];
  // (its barrier also publishes every warp's ranks and counters)
  int run = block_exclusive_base(mine, warp_tot_s);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int r = r_lo + j;
    if (j < ipt && r < R) {
      start_s[r] = run;
      run += cnt[j];
    }
  }
  if (threadIdx.x == kLayoutThreads - 1) start_s[R] = run;
  __syncthreads();
  const bool cap_ok = start_s[R] <= a.capacity;
  if (tile == 0 && threadIdx.x == 0 && !cap_ok) set_error(a.err, MOE_ERR_CAPACITY);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int r = threadIdx.x + j * kLayoutThreads;
    if (r < R && tile < T) {
      int b = start_s[r] + prior[j];
      for (int w = 0; w < kLayoutWarps; ++w) {
        const int c = cnt_s[w * R + r];
        cnt_s[w * R + r] = b;
        b += c;
      }
    }
  }
  __syncthreads();
  const int pairs_per_warp = plan.cpw * plan.lanes;
  const int npairs = tc.ntok * K;
  for (int i = threadIdx.x; i < npairs; i += blockDim.x) {
    const int e = ids_s[i];
    int slot = -1;
    if (e >= 0 && cap_ok && lr_s[i] >= 0) {
      slot = cnt_s[(i / pairs_per_warp) * R + e / L] + lr_s[i];
      a.rank_src[slot] = static_cast<int32_t>(tc.t0 + i / K);
    }
    a.rank_slot[tc.t0 * K + i] = slot;
  }
}

// Running per-expert totals across calls ([CS] §7.2: the receive statistics
// the page accumulates next to the alignment): cumulative[e] += count[e].
__global__ void __launch_bounds__(kLayoutThreads)
    accumulate_stats_kernel(const int32_t* __restrict__ expert_count, int E, int64_t* __restrict__ cumulative) {
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
    cumulative[e] += __ldcg(expert_count + e);
}

size_t fused_smem_bytes(const moe_layout_desc& d, const TilePlan& p) {
  const size_t pairs = static_cast<size_t>(p.tile_tokens) * d.topk;
  const size_t E = d.num_experts;
  return sizeof(int) * (2 * pairs + kLayoutWarps * E + 3 * E + 1 + d.num_ranks);
}

// Whether every tile's CTA of the fused kernel can be resident at once
// (device attribute and occupancy cached per device and size).
template <typename IdT>
bool fused_fits(const TilePlan& p, size_t smem) {
  if (p.tiles < 1 || !cooperative_launch_supported()) return false;
  const int per_sm = cached_occupancy(layout_fused_kernel<IdT>, kLayoutThreads, smem);
  return p.tiles <= static_cast<int64_t>(per_sm) * device_sm_count();
}

RankArgs rank_args(const moe_layout_desc& d, const int32_t* hist_prefix, const int32_t* expert_count,
                   const int32_t* rank_count, int32_t* expert_offset, int32_t* rank_psum, int32_t* dst_slot,
                   int32_t* src_idx, int64_t capacity, int32_t* total_rows, int* err) {
  RankArgs a;
  a.N = d.num_tokens;
  a.K = d.topk;
  a.E = d.num_experts;
  a.R = d.num_ranks;
  a.A = d.alignment;
  a.hist_prefix = hist_prefix;
  a.expert_count = expert_count;
  a.rank_count = rank_count;
  a.expert_offset = expert_offset;
  a.rank_psum = rank_psum;
  a.dst_slot = dst_slot;
  a.src_idx = src_idx;
  a.capacity = capacity;
  a.total_rows = total_rows;
  a.err = err;
  const WaitConfig wc = wait_config();
  a.wait_ns = wc.limit_ns;
  a.barrier_extra = wc.barrier_extra;
  return a;
}

}  // namespace

size_t count_smem_bytes(const moe_layout_desc& d, const TilePlan& p) {
  return sizeof(int) * (static_cast<size_t>(d.num_experts) + d.num_ranks +
                        static_cast<size_t>(p.tile_tokens) * d.topk);
}

size_t rank_smem_bytes(const moe_layout_desc& d, const TilePlan& p) {
  return sizeof(int) * (3 * static_cast<size_t>(d.num_experts) + 1 +
                        static_cast<size_t>(kLayoutWarps) * d.num_experts +
                        2 * static_cast<size_t>(p.tile_tokens) * d.topk);
}

namespace {

template <typename IdT>
cudaError_t launch_count_t(const moe_layout_desc& d, const TilePlan& p, const IdT* topk_idx, int32_t* expert_count,
                           int32_t* rank_count, int* err, int32_t* hist, int32_t* rhist, cudaStream_t stream) {
  const size_t smem1 = count_smem_bytes(d, p);
  cudaError_t st = ensure_smem_limit(count_tiles_kernel<IdT>, smem1);
  if (st != cudaSuccess) return st;
  if (p.tiles > 0) {
    st = launch_pdl(count_tiles_kernel<IdT>, dim3(static_cast<unsigned>(p.tiles)), dim3(kLayoutThreads), smem1,
                    stream, topk_idx, d.num_tokens, d.topk, d.num_experts, d.num_ranks, p, hist, rhist, err);
    if (st != cudaSuccess) return st;
    count_launch();
  }
  const int rows = d.num_experts + d.num_ranks;
  st = launch_pdl(scan_columns_kernel, dim3((rows + kLayoutWarps - 1) / kLayoutWarps), dim3(kLayoutThreads), 0,
                  stream, hist, rhist, p.tiles, d.num_experts, d.num_ranks, expert_count, rank_count);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

template <typename IdT>
cudaError_t launch_rank_t(const moe_layout_desc& d, const TilePlan& p, const IdT* topk_idx, const RankArgs& a,
                          cudaStream_t stream) {
  const size_t smem = rank_smem_bytes(d, p);
  cudaError_t st = ensure_smem_limit(rank_maps_kernel<IdT>, smem);
  if (st != cudaSuccess) return st;
  const int64_t grid = p.tiles > 0 ? p.tiles : 1;
  st = launch_pdl(rank_maps_kernel<IdT>, dim3(static_cast<unsigned>(grid)), dim3(kLayoutThreads), smem, stream,
                  topk_idx, p, a);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

template <typename IdT>
cudaError_t launch_rank_rows_t(const moe_layout_desc& d, const TilePlan& p, const IdT* topk_idx,
                               const RankRowsArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(int) * (static_cast<size_t>(d.num_ranks) + 1 +
                                     static_cast<size_t>(kLayoutWarps) * d.num_ranks +
                                     2 * static_cast<size_t>(p.tile_tokens) * d.topk);
  cudaError_t st = ensure_smem_limit(rank_rows_kernel<IdT>, smem);
  if (st != cudaSuccess) return st;
  const int64_t grid = p.tiles > 0 ? p.tiles : 1;
  st = launch_pdl(rank_rows_kernel<IdT>, dim3(static_cast<unsigned>(grid)), dim3(kLayoutThreads), smem, stream,
                  topk_idx, p, a);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

// Set once a driver has refused the cooperative + PDL launch pair; read by
// every later build, from any host thread.
std::atomic<bool>& fused_pdl_refused() {
  static std::atomic<bool> refused{false};
  return refused;
}

template <typename IdT>
cudaError_t launch_build_t(const moe_layout_desc& d, const TilePlan& p, const IdT* topk_idx, int32_t* expert_count,
                           int32_t* rank_count, int32_t* hist, int32_t* rhist, unsigned* barrier_words,
                           const RankArgs& a, cudaStream_t stream) {
  const size_t smem = fused_smem_bytes(d, p);
  // The three PDL-chained kernels rank each tile before the rank kernel's
  // wait, overlapping the count and the column scan; the cooperative kernel
  // does the phases one after another but saves two launches.  Measured on
  // GB300 (one-call layout, top-8; chained / cooperative): 16384 tokens 13.8 /
  // 16.5 us, 65536 21.8 / 22.1, 98304 25.7 / 26.6, 131072 (16 chunks per
  // warp) 31.2 / 30.4.  So the cooperative kernel runs only when a tile holds
  // the most chunks per warp and every tile's CTA fits on the GPU at once.
  if (p.cpw < kMaxChunksPerWarp || !fused_fits<IdT>(p, smem)) {
    cudaError_t st = launch_count_t(d, p, topk_idx, expert_count, rank_count, a.err, hist, rhist, stream);
    if (st != cudaSuccess) return st;
    return launch_rank_t(d, p, topk_idx, a, stream);
  }
  if (cudaError_t st = ensure_smem_limit(layout_fused_kernel<IdT>, smem)) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.tiles));
  cfg.blockDim = dim3(kLayoutThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // Cooperative, and allowed to start during the previous kernel's tail (it
  // waits with griddepcontrol.wait before reading anything).  A driver that
  // refuses the pair gets the plain cooperative launch.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = fused_pdl_refused().load(std::memory_order_relaxed) ? 1 : 2;
  cudaError_t st = cudaLaunchKernelEx(&cfg, layout_fused_kernel<IdT>, topk_idx, p, a, hist, rhist, expert_count,
                                      rank_count, barrier_words);
  if (st != cudaSuccess && cfg.numAttrs == 2) {
    (void)cudaGetLastError();
    fused_pdl_refused().store(true, std::memory_order_relaxed);
    cfg.numAttrs = 1;
    st = cudaLaunchKernelEx(&cfg, layout_fused_kernel<IdT>, topk_idx, p, a, hist, rhist, expert_count, rank_count,
                            barrier_words);
  }
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_count(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, int32_t* expert_count,
                         int32_t* rank_count, int* err, int32_t* hist, int32_t* rhist, cudaStream_t stream) {
  return ids.i32 ? launch_count_t(d, p, static_cast<const int32_t*>(ids.ptr), expert_count, rank_count, err, hist,
                                  rhist, stream)
                 : launch_count_t(d, p, static_cast<const int64_t*>(ids.ptr), expert_count, rank_count, err, hist,
                                  rhist, stream);
}

cudaError_t launch_rank(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, const int32_t* hist_prefix,
                        const int32_t* expert_count, const int32_t* rank_count, int32_t* expert_offset,
                        int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx, int64_t capacity,
                        int32_t* total_rows, int* err, cudaStream_t stream) {
  const RankArgs a = rank_args(d, hist_prefix, expert_count, rank_count, expert_offset, rank_psum, dst_slot,
                               src_idx, capacity, total_rows, err);
  return ids.i32 ? launch_rank_t(d, p, static_cast<const int32_t*>(ids.ptr), a, stream)
                 : launch_rank_t(d, p, static_cast<const int64_t*>(ids.ptr), a, stream);
}

cudaError_t launch_accumulate_stats(const int32_t* expert_count, int E, int64_t* cumulative, cudaStream_t stream) {
  const cudaError_t st = launch_pdl(accumulate_stats_kernel, dim3((E + kLayoutThreads - 1) / kLayoutThreads),
                                    dim3(kLayoutThreads), 0, stream, expert_count, E, cumulative);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_rank_rows(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, const int32_t* rhist_prefix,
                             const int32_t* rank_count, int32_t* rank_slot, int32_t* rank_src, int64_t capacity,
                             int* err, cudaStream_t stream) {
  RankRowsArgs a;
  a.N = d.num_tokens;
  a.K = d.topk;
  a.E = d.num_experts;
  a.R = d.num_ranks;
  a.rhist_prefix = rhist_prefix;
  a.rank_count = rank_count;
  a.rank_slot = rank_slot;
  a.rank_src = rank_src;
  a.capacity = capacity;
  a.err = err;
  return ids.i32 ? launch_rank_rows_t(d, p, static_cast<const int32_t*>(ids.ptr), a, stream)
                 : launch_rank_rows_t(d, p, static_cast<const int64_t*>(ids.ptr), a, stream);
}

cudaError_t launch_build(const moe_layout_desc& d, const TilePlan& p, IdsRef ids, int32_t* expert_count,
                         int32_t* rank_count, int32_t* hist, int32_t* rhist, unsigned* barrier_words,
                         int32_t* expert_offset, int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx,
                         int64_t capacity, int32_t* total_rows, int* err, cudaStream_t stream) {
  const RankArgs a = rank_args(d, hist, expert_count, rank_count, expert_offset, rank_psum, dst_slot, src_idx,
                               capacity, total_rows, err);
  return ids.i32 ? launch_build_t(d, p, static_cast<const int32_t*>(ids.ptr), expert_count, rank_count, hist, rhist,
                                  barrier_words, a, stream)
                 : launch_build_t(d, p, static_cast<const int64_t*>(ids.ptr), expert_count, rank_count, hist, rhist,
                                  barrier_words, a, stream);
}

}  // namespace moe
