// combine_kernel.cu -- inverse of the dispatch on sm_103a: gather each
// token's expert-output rows through dst_slot and reduce them with the
// token's top-k weights.
//
//   out[t, h] = bf16_rn( fma(w[t,K-1], y[K-1], ... fma(w[t,0], y[0], 0.0f)) )
//   with y[k] = float(expert_out[dst_slot[t,k], h]), masked k skipped.
//
// The page "07 DeepEP Counting Sort / Bucketization" keeps the slot map for
// the combine (§6.2) but prints no combine arithmetic; the order above (fp32
// from 0, ascending k, one fused multiply-add per term, one bf16 rounding) is
// the plain definition and makes the result bit-reproducible.
//
// HBM-bound.  Two kernels, chosen by batch size:
//  - combine_bulk_kernel (from 12 tokens per resident CTA): a persistent
//    grid whose producer warps move each token's expert rows into a shared-
//    memory ring with bulk copies while consumer warps run the fma chain out
//    of shared memory (its own section below);
//  - combine_kernel (smaller batches): each thread owns 16-byte column
//    vectors of the row and issues the loads of up to 8 expert rows before any
//    arithmetic, so 8 x 16 B per thread are in flight; slots and weights of the
//    CTA's token block are staged in shared memory once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Grid = whole waves at the kernel's occupancy, tokens shared out evenly over
// exactly that many CTAs (a grid of 1.7 waves left a third of the SMs idle
// during the partial second wave).  Small batches get more, smaller CTAs for
// the block scheduler to balance: measured on GB300, 4 waves took decode's
// combine from 90.5 to 88.2 us, while 131072 tokens ran 1 % faster with 2.
#ifndef MOE_COMBINE_WAVES
#define MOE_COMBINE_WAVES 2
#endif
#ifndef MOE_COMBINE_SMALL_WAVES
#define MOE_COMBINE_SMALL_WAVES 4
#endif
#ifndef MOE_COMBINE_SMALL_TOKENS_PER_CTA
#define MOE_COMBINE_SMALL_TOKENS_PER_CTA 8   // "small": fewer tokens per CTA than this at SMALL_WAVES
#endif

constexpr int kCombineThreads = 256;
constexpr int kKGroup = 8;              // expert rows loaded before their FMAs
constexpr int kMaxTokensPerCta = 64;
#ifndef MOE_COMBINE_VEC_UNROLL
#define MOE_COMBINE_VEC_UNROLL 1
#endif
constexpr int kVecUnroll = MOE_COMBINE_VEC_UNROLL;

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fmaf_rn(w, __uint_as_float(u[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// CTA b's share of n items split over g CTAs: [share_start(b), share_start(b + 1)).
__device__ __forceinline__ int64_t share_start(int64_t b, int64_t n, int64_t g) {
  return b * (n / g) + min64(b, n % g);
}

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const CombineArgs a, int max_tokens) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = a.topk;
  int32_t* slot_s = reinterpret_cast<int32_t*>(smem);
  float* w_s = reinterpret_cast<float*>(smem + sizeof(int32_t) * max_tokens * K);

  const int64_t t0 = share_start(blockIdx.x, a.num_tokens, gridDim.x);
  const int ntok = static_cast<int>(share_start(static_cast<int64_t>(blockIdx.x) + 1, a.num_tokens, gridDim.x) - t0);
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  // Slots and weights of the CTA's tokens; kBatch independent loads of each per thread.
  constexpr int kBatch = 4;
  for (int base = threadIdx.x; base < ntok * K; base += kBatch * kCombineThreads) {
    int sv[kBatch];
    float wv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kCombineThreads;
      const bool in = i < ntok * K;
      sv[u] = in ? __ldg(a.dst_slot + t0 * K + i) : -1;
      wv[u] = in ? __ldg(a.weights + t0 * K + i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kCombineThreads;
      if (i >= ntok * K) break;
      int s = sv[u];
      if (s >= a.expert_out_rows) {
        set_error(a.err, MOE_ERR_CAPACITY);
        s = -1;
      }
      slot_s[i] = s;
      w_s[i] = wv[u];
    }
  }
  __syncthreads();

  const int64_t H = a.hidden;
  const int nvec = static_cast<int>(H / 8);
  for (int tt = 0; tt < ntok; ++tt) {
    const int32_t* sl = slot_s + tt * K;
    const float* wt = w_s + tt * K;
    uint16_t* orow = a.out + (t0 + tt) * H;
    // kVecUnroll column vectors per thread per pass, all their row loads in
    // flight before the FMAs.
    for (int j0 = threadIdx.x; j0 < nvec; j0 += kVecUnroll * kCombineThreads) {
      float acc[kVecUnroll][8];
#pragma unroll
      for (int x = 0; x < kVecUnroll; ++x)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[x][i] = 0.0f;
      for (int kg = 0; kg < K; kg += kKGroup) {
        uint4 v[kVecUnroll][kKGroup];
#pragma unroll
        for (int x = 0; x < kVecUnroll; ++x) {
          const int j = j0 + x * kCombineThreads;
#pragma unroll
          for (int q = 0; q < kKGroup; ++q) {
            const int k = kg + q;
            const int32_t s = (k < K && j < nvec) ? sl[k] : -1;
            v[x][q] = s >= 0 ? ptx::ld_nc_v4(a.expert_out + static_cast<int64_t>(s) * H + j * 8)
                             : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int x = 0; x < kVecUnroll; ++x)
#pragma unroll
          for (int q = 0; q < kKGroup; ++q) {
            const int k = kg + q;
            if (k < K && sl[k] >= 0) fma_bf16x8(acc[x], wt[k], v[x][q]);
          }
      }
#pragma unroll
      for (int x = 0; x < kVecUnroll; ++x) {
        const int j = j0 + x * kCombineThreads;
        if (j >= nvec) break;
        uint4 o;
        o.x = pack_bf16x2(acc[x][0], acc[x][1]);
        o.y = pack_bf16x2(acc[x][2], acc[x][3]);
        o.z = pack_bf16x2(acc[x][4], acc[x][5]);
        o.w = pack_bf16x2(acc[x][6], acc[x][7]);
        ptx::st_v4(orow + j * 8, o);
      }
    }
  }
}

// ------------------------------------------------------ bulk-copy combine
// Batches of 12 or more tokens per resident CTA.  A persistent grid; in each
// CTA one producer warp takes tokens (its first two fixed, the rest claimed
// from a counter in the workspace, three tokens in flight) and
// moves the token's expert rows, a piece of the row at a time, into a ring of
// shared-memory stages with bulk copies (cp.async.bulk, completion on the
// stage's mbarrier): lane k copies row k, so the K copies of a piece go out
// together and one warp keeps a whole ring of rows in flight without holding
// any of it in registers.  Two groups of four consumer warps take the stages
// in turn: each thread reads the K rows' 16-byte column vector from shared
// memory, runs the fma chain in ascending k and stores the bf16 result.
// Each stage starts with a header (token, piece, valid-row mask, weights)
// that the producer writes before it arms the stage.
#ifndef MOE_COMBINE_BULK
#define MOE_COMBINE_BULK 1
#endif
// Ring budget and CTAs per SM, measured on GB300 (combine time, round-trip /
// skewed / decode workloads): 3 CTAs of 4 stages (70 KB) 1309 / 285 / 90 us;
// 2 CTAs of 6 stages (100 KB) 1348 / 287 / 89 us; 1 CTA of 12 stages (200 KB)
// 2402 / 492 / 135 us, a CTA's stages turning over no faster than ~0.7 us
// each whatever the depth, so the SM needs several CTAs.
#ifndef MOE_COMBINE_BULK_RING_BYTES
#define MOE_COMBINE_BULK_RING_BYTES 70000
#endif
#ifndef MOE_COMBINE_BULK_CTAS_PER_SM
#define MOE_COMBINE_BULK_CTAS_PER_SM 3
#endif
// Batches with fewer tokens than this per resident CTA of the bulk kernel
// take the register kernel instead (decode: 4096 tokens, 9 per CTA, combine
// 88 us there against 90 us in the bulk kernel, whose tail is a whole token
// of a CTA's ring).
#ifndef MOE_COMBINE_BULK_MIN_TOKENS_PER_CTA
#define MOE_COMBINE_BULK_MIN_TOKENS_PER_CTA 12
#endif
#ifndef MOE_COMBINE_PIECE_BYTES
#define MOE_COMBINE_PIECE_BYTES 16384   // target bytes of one stage's rows (K pieces)
#endif
constexpr int kBulkGroupThreads = 128;   // consumer threads per group: one 16-byte column vector each
constexpr int kBulkGroups = 2;
constexpr int kBulkGroupWarps = kBulkGroupThreads / kWarpSize;
constexpr int kBulkThreads = kWarpSize + kBulkGroups * kBulkGroupThreads;
constexpr int kBulkMaxStages = 16;
constexpr int kStageHeaderBytes = 256;
constexpr int kMaxPieceCols = 8 * kBulkGroupThreads;   // 1024 columns

struct StageHeader {
  int64_t token;    // -1: no more stages for the consumer group that takes this one
  int32_t piece;
  uint32_t valid;   // bit k: the stage holds expert row k of the token
  float w[MOE_MAX_TOPK];
};
static_assert(sizeof(StageHeader) <= kStageHeaderBytes, "stage header");

struct BulkPlan {
  int piece_cols;    // columns per piece: a multiple of 8, at most kMaxPieceCols
  int pieces;        // pieces per row; the last may be shorter
  int stage_bytes;   // header + K piece rows, a multiple of 128
  int stages;
};

__global__ void __launch_bounds__(kBulkThreads, 1)
    combine_bulk_kernel(const CombineArgs a, const BulkPlan p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kBulkMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kBulkMaxStages];
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int K = a.topk, S = p.stages, PC = p.piece_cols;
  const int64_t H = a.hidden, N = a.num_tokens;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], kBulkGroupWarps);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();

  if (warp == 0) {
    // ---- producer warp -----------------------------------------------------
    unsigned* next_tok = a.work;
    unsigned* done_ctas = a.work + 1;
    const unsigned kFull = 0xffffffffu;
    const uint64_t policy = ptx::l2_evict_first_policy();   // each expert row is read once
    // Lane 0 issues the claim; its value is broadcast only when it is needed,
    // so the atomic's latency overlaps the work in between.
    // Each CTA's first two tokens are fixed (blockIdx.x and blockIdx.x + G);
    // the rest are claimed from the counter (claim c is token 2G + c).
    const int64_t G = gridDim.x;
    auto claim = [&]() -> unsigned { return lane == 0 ? atomicAdd(next_tok, 1u) : 0u; };
    auto broadcast = [&](unsigned v) -> int64_t { return 2 * G + static_cast<int64_t>(__shfl_sync(kFull, v, 0)); };
    // A three-token pipeline, so that neither a claim's atomic nor the slot
    // loads that depend on it stall the copies.  Three register sets rotate
    // through the roles (issued now / loading / claimed) without being copied:
    // a copy of a register whose load is still in flight would wait for it.
    // In each phase token A is issued (its slots and weights, lane k holding
    // pair k, were loaded two phases ago), C's claim is broadcast and its
    // slots are requested, and the next claim goes out.
    int64_t t0 = blockIdx.x, t1 = blockIdx.x + G, t2 = 0;
    int32_t s0 = -1, s1 = -1, s2 = -1;
    float w0 = 0.0f, w1 = 0.0f, w2 = 0.0f;
    unsigned pending = claim();
    if (t0 < N && lane < K) {
      s0 = __ldg(a.dst_slot + t0 * K + lane);
      w0 = __ldg(a.weights + t0 * K + lane);
    }
    if (t1 < N && lane < K) {
      s1 = __ldg(a.dst_slot + t1 * K + lane);
      w1 = __ldg(a.weights + t1 * K + lane);
    }
    int64_t j = 0;   // stages armed so far (stage j % S, its use j / S)
    bool ok = true;
    auto acquire_stage = [&](int64_t jj) -> bool {
      const int s = static_cast<int>(jj % S);
      const int64_t use = jj / S;
      bool got = true;
      if (use > 0 && lane == 0)
        got = ptx::mbar_wait_parity_bounded(&empty_bar[s], static_cast<uint32_t>((use - 1) & 1), a.wait_ns);
      return __shfl_sync(kFull, got ? 1 : 0, 0) != 0;
    };
    // One phase; false once token A is past the end (or a wait ran out).
    auto phase = [&](const int64_t tA, const int32_t sA, const float wA, int64_t& tC, int32_t& sC,
                     float& wC) -> bool {
      if (tA >= N) return false;
      const unsigned next = claim();
      tC = broadcast(pending);
      pending = next;
      if (tC < N && lane < K) {
        sC = __ldg(a.dst_slot + tC * K + lane);
        wC = __ldg(a.weights + tC * K + lane);
      }
      bool valid = false;
      if (lane < K && sA >= 0) {
        if (sA < a.expert_out_rows)
          valid = true;
        else
          set_error(a.err, MOE_ERR_CAPACITY);
      }
      const unsigned mask = __ballot_sync(kFull, valid);
      for (int c = 0; c < p.pieces; ++c, ++j) {
        if (!acquire_stage(j)) {
          ok = false;
          return false;
        }
        const int s = static_cast<int>(j % S);
        uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
        StageHeader* h = reinterpret_cast<StageHeader*>(st);
        const int64_t col0 = static_cast<int64_t>(c) * PC;
        const uint32_t bytes = static_cast<uint32_t>(min64(PC, H - col0) * 2);
        if (lane < K) h->w[lane] = wA;
        if (lane == 0) {
          h->token = tA;
          h->piece = c;
          h->valid = mask;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_expect_tx(&full_bar[s], bytes * static_cast<uint32_t>(__popc(mask)));
        __syncwarp();
        if (valid)
          ptx::bulk_g2s_hint(st + kStageHeaderBytes + static_cast<size_t>(lane) * PC * 2,
                             a.expert_out + static_cast<int64_t>(sA) * H + col0, bytes, &full_bar[s], policy);
      }
      return true;
    };
    while (phase(t0, s0, w0, t2, s2, w2) && phase(t1, s1, w1, t0, s0, w0) && phase(t2, s2, w2, t1, s1, w1)) {
    }
    // One end marker for each consumer group.
    for (int g = 0; g < kBulkGroups && ok; ++g, ++j) {
      if (!acquire_stage(j)) {
        ok = false;
        break;
      }
      const int s = static_cast<int>(j % S);
      if (lane == 0) {
        reinterpret_cast<StageHeader*>(smem + static_cast<size_t>(s) * p.stage_bytes)->token = -1;
        ptx::mbar_arrive(&full_bar[s]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (!ok) {
        set_error(a.err, MOE_ERR_TIMEOUT);
        // Let every copy already issued land before the CTA's shared memory goes away:
        // the last arming of each stage (earlier ones completed before it was reused).
        for (int64_t v = max64(0, j - S); v < j; ++v)
          ptx::mbar_wait_parity_bounded(&full_bar[v % S], static_cast<uint32_t>((v / S) & 1), a.wait_ns);
      }
      // The last CTA to finish claiming resets both counters for the next launch.
      __threadfence();
      if (atomicAdd(done_ctas, 1u) == gridDim.x - 1) {
        atomicExch(next_tok, 0u);
        atomicExch(done_ctas, 0u);
      }
    }
    return;
  }

  // ---- consumer groups: stages g, g + 2, g + 4, ... --------------------------
  const int g = (warp - 1) / kBulkGroupWarps;
  const int ct = threadIdx.x - kWarpSize - g * kBulkGroupThreads;
  for (int64_t j = g;; j += kBulkGroups) {
    const int s = static_cast<int>(j % S);
    if (!ptx::mbar_wait_parity_bounded(&full_bar[s], static_cast<uint32_t>((j / S) & 1), a.wait_ns)) {
      set_error(a.err, MOE_ERR_TIMEOUT);
      return;
    }
    const uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
    const StageHeader* h = reinterpret_cast<const StageHeader*>(st);
    const int64_t token = h->token;
    if (token < 0) return;
    const int64_t col0 = static_cast<int64_t>(h->piece) * PC;
    const unsigned mask = h->valid;
    const int64_t ncol = min64(PC, H - col0);
    if (ct * 8 < ncol) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      const uint8_t* rows = st + kStageHeaderBytes + ct * 16;
      for (int k = 0; k < K; ++k) {
        if ((mask >> k) & 1u) fma_bf16x8(acc, h->w[k], ptx::ld_shared_v4(rows + static_cast<size_t>(k) * PC * 2));
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      ptx::st_v4(a.out + token * H + col0 + ct * 8, o);
    }
    // Every lane's shared-memory reads of the stage completed before its
    // store (which uses them).  The arrival is relaxed: a releasing one would
    // wait for the stores to reach memory first, a round trip per stage.
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_relaxed(&empty_bar[s]);
  }
}

BulkPlan make_bulk_plan(const CombineArgs& a) {
  BulkPlan p{};
  int pc = static_cast<int>(MOE_COMBINE_PIECE_BYTES / (2 * a.topk)) / 8 * 8;
  pc = std::max(8, std::min(kMaxPieceCols, pc));
  p.piece_cols = static_cast<int>(min64(pc, a.hidden));
  p.pieces = static_cast<int>(ceil_div64(a.hidden, p.piece_cols));
  p.stage_bytes = (kStageHeaderBytes + a.topk * p.piece_cols * 2 + 127) / 128 * 128;
  // An even number of stages: stage s then always feeds consumer group s % 2,
  // which waits on its uses in order.  (With an odd count the two groups
  // would alternate on one stage, and a group could wait for a use before the
  // other group's earlier use completed: an mbarrier wait only tells parity.)
  p.stages = std::max(2, std::min(kBulkMaxStages, MOE_COMBINE_BULK_RING_BYTES / p.stage_bytes)) & ~1;
  return p;
}

// Resident CTAs per SM at the largest shared-memory size a launch uses (cached per device).
int combine_ctas_per_sm() {
  const size_t smem = (sizeof(int32_t) + sizeof(float)) * kMaxTokensPerCta * MOE_MAX_TOPK;
  const int occ = cached_occupancy(combine_kernel, kCombineThreads, smem);
  return occ < 1 ? 1 : occ;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& args, cudaStream_t stream) {
  CombineArgs a = args;
  a.wait_ns = wait_config().limit_ns;
  // Claims run to at most N + 2 * grid, inside the 32-bit counter (N * K < 2^31).
  const BulkPlan bp = make_bulk_plan(a);
  const size_t bulk_smem = static_cast<size_t>(bp.stages) * bp.stage_bytes;
  int per_sm = cached_occupancy(combine_bulk_kernel, kBulkThreads, bulk_smem);
  if (per_sm < 1) per_sm = 1;
  if (MOE_COMBINE_BULK_CTAS_PER_SM > 0 && MOE_COMBINE_BULK_CTAS_PER_SM < per_sm) per_sm = MOE_COMBINE_BULK_CTAS_PER_SM;
  const int64_t bulk_resident = static_cast<int64_t>(per_sm) * device_sm_count();
  if (MOE_COMBINE_BULK && a.work != nullptr &&
      a.num_tokens >= static_cast<int64_t>(MOE_COMBINE_BULK_MIN_TOKENS_PER_CTA) * bulk_resident) {
    const BulkPlan& p = bp;
    const size_t smem = bulk_smem;
    if (cudaError_t st = ensure_smem_limit(combine_bulk_kernel, smem)) return st;
    const int64_t grid = max64(1, min64(bulk_resident, a.num_tokens));
    const cudaError_t st =
        launch_pdl(combine_bulk_kernel, dim3(static_cast<unsigned>(grid)), dim3(kBulkThreads), smem, stream, a, p);
    if (st != cudaSuccess) return st;
    count_launch();
    return cudaSuccess;
  }
  const int64_t resident = static_cast<int64_t>(combine_ctas_per_sm()) * device_sm_count();
  const bool small = a.num_tokens < static_cast<int64_t>(MOE_COMBINE_SMALL_TOKENS_PER_CTA) * MOE_COMBINE_SMALL_WAVES * resident;
  // Whole waves, each CTA at least one token and at most kMaxTokensPerCta
  // (shared out evenly: counts differ by at most one).
  int64_t grid = (small ? MOE_COMBINE_SMALL_WAVES : MOE_COMBINE_WAVES) * resident;
  grid = max64(grid, ceil_div64(a.num_tokens, kMaxTokensPerCta));
  grid = max64(1, min64(grid, a.num_tokens));
  const int64_t max_tokens = max64(1, ceil_div64(a.num_tokens, grid));
  const size_t smem = (sizeof(int32_t) + sizeof(float)) * static_cast<size_t>(max_tokens) * a.topk;
  // Small batches start during the previous kernel's tail (programmatic
  // dependent launch); large ones start after it: measured on GB300, the
  // overlap saved 1.2 us of a decode step and cost 26 us of a 131072-token one.
  // Both go through cudaLaunchKernelEx, whose status is this launch's own
  // (an error left over from an earlier runtime call is not picked up).
  const cudaError_t st = small ? launch_pdl(combine_kernel, dim3(static_cast<unsigned>(grid)), dim3(kCombineThreads),
                                            smem, stream, a, static_cast<int>(max_tokens))
                               : launch_plain(combine_kernel, dim3(static_cast<unsigned>(grid)),
                                              dim3(kCombineThreads), smem, stream, a, static_cast<int>(max_tokens));
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
