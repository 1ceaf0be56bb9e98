// permute_kernel.cu -- expand-mode dispatch permute on sm_103a: every valid
// (token, k) copy of a row goes to its slot in the expert-major receive
// buffer, and the alignment-gap rows are zeroed.
//
// Method: page "07 DeepEP Counting Sort / Bucketization", §6.3-§6.4 (rows
// moved by 1-D TMA stores to their slot), §7.3 (zero padding), §8.2 (expand
// mode).  The page moves rows twice (rank buffer, then expert buffer) across
// GPUs; with logical ranks on one GPU the expert-major buffer is written
// directly, once.
//
// Design (HBM-bound, no arithmetic):
//  - token-major: each token row is read from HBM once into shared memory by
//    a bulk copy (cp.async.bulk, completion on an mbarrier) and written K
//    times by bulk shared->global stores, so reads are N rows, not N*K;
//  - one elected thread per CTA drives a multi-stage shared-memory ring, so
//    several row loads are in flight while earlier rows are stored;
//  - the CTA's other warps zero its share of the gap rows with 16-byte
//    stores and move the (small, 4-byte aligned) scale-factor rows;
//  - gap rows are split evenly over CTAs by a prefix sum of gap sizes, so a
//    hot expert with a big gap does not land on one CTA.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

#ifndef MOE_PERMUTE_CTAS_PER_SM
#define MOE_PERMUTE_CTAS_PER_SM 4
#endif
#ifndef MOE_PERMUTE_STAGE_BUDGET
#define MOE_PERMUTE_STAGE_BUDGET (48 * 1024)
#endif

constexpr int kPermuteThreads = 256;
constexpr int kPermuteWarps = kPermuteThreads / kWarpSize;
constexpr int kMaxStages = 8;
constexpr int kMaxChunkBytes = 16384;
constexpr int kStageBudgetBytes = MOE_PERMUTE_STAGE_BUDGET;  // shared-memory ring per CTA
constexpr int kCtasPerSm = MOE_PERMUTE_CTAS_PER_SM;           // grid sizing target
constexpr int kMaxTokensPerCta = 512;
constexpr int kSfRegWords = 4;  // scale-factor words a lane keeps in registers

struct PermutePlan {
  int chunk_bytes;     // bytes per bulk load (a row, or a 16 KiB slice of it)
  int nchunks;         // slices per row
  int stages;          // shared-memory ring depth
  int tokens_per_cta;
  int64_t grid;
  size_t off_slots, off_active, off_padpre, smem;
};

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < kWarpSize; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

// padpre[e] = sum over e' < e of the gap rows of expert e' (E+1 entries).
__device__ void gap_prefix(const int32_t* __restrict__ off, const int32_t* __restrict__ cnt, int E,
                           int32_t* padpre, int* warp_tot) {
  const int lane = threadIdx.x % kWarpSize, warp = threadIdx.x / kWarpSize;
  const int ipt = (E + kPermuteThreads - 1) / kPermuteThreads;
  const int e_lo = threadIdx.x * ipt;
  int mine = 0;
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) mine += __ldg(off + e + 1) - __ldg(off + e) - __ldg(cnt + e);
  }
  const int incl = warp_inclusive_scan(mine, lane);
  if (lane == kWarpSize - 1) warp_tot[warp] = incl;
  __syncthreads();
  int run = incl - mine;
  for (int w = 0; w < warp; ++w) run += warp_tot[w];
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) {
      padpre[e] = run;
      run += __ldg(off + e + 1) - __ldg(off + e) - __ldg(cnt + e);
    }
  }
  if (threadIdx.x == kPermuteThreads - 1) padpre[E] = run;
}

__global__ void __launch_bounds__(kPermuteThreads)
    permute_kernel(const PermuteArgs a, const PermutePlan p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ int warp_tot_s[kPermuteWarps];
  uint8_t* ring = smem;
  int32_t* slots_s = reinterpret_cast<int32_t*>(smem + p.off_slots);
  int32_t* active_s = reinterpret_cast<int32_t*>(smem + p.off_active);
  int32_t* padpre_s = reinterpret_cast<int32_t*>(smem + p.off_padpre);

  const int K = a.topk, E = a.num_experts;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * p.tokens_per_cta;
  const int ntok = static_cast<int>(max64(0, min64(p.tokens_per_cta, a.num_tokens - t0)));
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) ptx::mbar_init(&full_bar[s], 1);
    ptx::fence_mbar_init();
  }
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  const int64_t rows = __ldg(a.total_rows);
  if (rows > a.capacity) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, MOE_ERR_CAPACITY);
    return;
  }

  for (int i = threadIdx.x; i < ntok * K; i += kPermuteThreads) {
    int s = __ldg(a.dst_slot + t0 * K + i);
    if (s >= a.capacity) {
      set_error(a.err, MOE_ERR_CAPACITY);
      s = -1;
    }
    slots_s[i] = s;
  }
  if (a.zero_pad) gap_prefix(a.expert_offset, a.expert_count, E, padpre_s, warp_tot_s);
  __syncthreads();

  if (warp == 0) {
    // Tokens with at least one valid slot, in order.
    int n_active = 0;
    for (int base = 0; base < ntok; base += kWarpSize) {
      const int tok = base + lane;
      bool act = false;
      if (tok < ntok)
        for (int k = 0; k < K; ++k) act |= slots_s[tok * K + k] >= 0;
      const unsigned b = __ballot_sync(0xffffffffu, act);
      if (act) active_s[n_active + __popc(b & ptx::lanemask_lt())] = tok;
      n_active += __popc(b);
    }
    __syncwarp();
    if (lane != 0) return;

    // ---- producer: one thread drives the bulk-copy ring -------------------
    const int64_t rb = a.row_bytes;
    const int chunk = p.chunk_bytes, S = p.stages, nch = p.nchunks;
    const int units = n_active * nch;
    auto unit_bytes = [&](int c) -> uint32_t {
      return static_cast<uint32_t>(min64(chunk, rb - static_cast<int64_t>(c) * chunk));
    };
    auto issue = [&](int u) {
      const int s = u % S, tok = active_s[u / nch], c = u % nch;
      const uint32_t bytes = unit_bytes(c);
      ptx::mbar_arrive_expect_tx(&full_bar[s], bytes);
      ptx::bulk_g2s(ring + static_cast<size_t>(s) * chunk,
                    a.x + (t0 + tok) * rb + static_cast<int64_t>(c) * chunk, bytes, &full_bar[s]);
    };
    const int prologue = min(S, units);
    for (int u = 0; u < prologue; ++u) issue(u);
    int u = 0;
    bool ok = true;
    for (; u < units; ++u) {
      const int s = u % S;
      if (!ptx::mbar_wait_parity_bounded(&full_bar[s], (u / S) & 1, kWaitLimitNs)) {
        ok = false;
        break;
      }
      const int tok = active_s[u / nch], c = u % nch;
      const uint32_t bytes = unit_bytes(c);
      const int32_t* sl = slots_s + tok * K;
      const uint8_t* src = ring + static_cast<size_t>(s) * chunk;
      for (int k = 0; k < K; ++k) {
        const int32_t slot = sl[k];
        if (slot >= 0) ptx::bulk_s2g(a.recv_x + slot * rb + static_cast<int64_t>(c) * chunk, src, bytes);
      }
      ptx::bulk_commit();
      if (u + S < units) {
        ptx::bulk_wait_read<0>();  // this stage's stores have read it
        issue(u + S);
      }
    }
    if (!ok) {
      set_error(a.err, MOE_ERR_TIMEOUT);
      // Let the loads already issued land before the CTA's shared memory goes away.
      for (int v = u; v < min(u + S, units); ++v)
        ptx::mbar_wait_parity_bounded(&full_bar[v % S], (v / S) & 1, kWaitLimitNs);
    }
    ptx::bulk_wait<0>();
    return;
  }

  // ---- helper warps: gap rows and scale-factor rows ------------------------
  const int htid = threadIdx.x - kWarpSize;
  const int nhelp = kPermuteThreads - kWarpSize;
  const int hwarp = warp - 1, nhwarps = kPermuteWarps - 1;

  if (a.zero_pad) {
    const int64_t total_pad = padpre_s[E];
    const int64_t G = gridDim.x;
    const int64_t p0 = total_pad * blockIdx.x / G, p1 = total_pad * (blockIdx.x + 1) / G;
    if (p0 < p1) {
      // First expert whose gap holds pad index p0.
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (padpre_s[mid] <= p0) lo = mid; else hi = mid - 1;
      }
      const uint4 zero = make_uint4(0, 0, 0, 0);
      for (int e = lo; e < E && padpre_s[e] < p1; ++e) {
        const int64_t a0 = max64(p0, padpre_s[e]), a1 = min64(p1, padpre_s[e + 1]);
        if (a0 >= a1) continue;
        const int64_t row0 = __ldg(a.expert_offset + e) + __ldg(a.expert_count + e) + (a0 - padpre_s[e]);
        const int64_t nrows = a1 - a0;
        uint8_t* base = a.recv_x + row0 * a.row_bytes;
        const int64_t n16 = nrows * a.row_bytes / 16;
        for (int64_t j = htid; j < n16; j += nhelp) ptx::st_cs_v4(base + j * 16, zero);
        if (a.recv_sf) {
          uint32_t* sb = reinterpret_cast<uint32_t*>(a.recv_sf + row0 * a.sf_row_bytes);
          const int64_t nw = nrows * a.sf_row_bytes / 4;
          for (int64_t j = htid; j < nw; j += nhelp) sb[j] = 0u;
        }
      }
    }
  }

  if (a.sf) {
    const int words = static_cast<int>(a.sf_row_bytes / 4);
    for (int tok = hwarp; tok < ntok; tok += nhwarps) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(a.sf + (t0 + tok) * a.sf_row_bytes);
      const int32_t* sl = slots_s + tok * K;
      if (words <= kSfRegWords * kWarpSize) {
        uint32_t v[kSfRegWords];
#pragma unroll
        for (int j = 0; j < kSfRegWords; ++j) {
          const int w = lane + j * kWarpSize;
          v[j] = w < words ? __ldg(src + w) : 0u;
        }
        for (int k = 0; k < K; ++k) {
          if (sl[k] < 0) continue;
          uint32_t* dst = reinterpret_cast<uint32_t*>(a.recv_sf + static_cast<int64_t>(sl[k]) * a.sf_row_bytes);
#pragma unroll
          for (int j = 0; j < kSfRegWords; ++j) {
            const int w = lane + j * kWarpSize;
            if (w < words) dst[w] = v[j];
          }
        }
      } else {
        for (int k = 0; k < K; ++k) {
          if (sl[k] < 0) continue;
          uint32_t* dst = reinterpret_cast<uint32_t*>(a.recv_sf + static_cast<int64_t>(sl[k]) * a.sf_row_bytes);
          for (int w = lane; w < words; w += kWarpSize) dst[w] = __ldg(src + w);
        }
      }
    }
  }
}

PermutePlan make_permute_plan(const PermuteArgs& a, int sms) {
  PermutePlan p{};
  p.chunk_bytes = static_cast<int>(min64(a.row_bytes, kMaxChunkBytes));
  p.nchunks = static_cast<int>(ceil_div64(a.row_bytes, p.chunk_bytes));
  p.stages = std::max(2, std::min(kMaxStages, kStageBudgetBytes / p.chunk_bytes));
  const int64_t target_ctas = static_cast<int64_t>(kCtasPerSm) * sms;
  int64_t tpc = ceil_div64(max64(a.num_tokens, 1), target_ctas);
  tpc = max64(1, min64(tpc, kMaxTokensPerCta));
  p.tokens_per_cta = static_cast<int>(tpc);
  p.grid = max64(1, ceil_div64(a.num_tokens, tpc));
  size_t off = static_cast<size_t>(p.stages) * p.chunk_bytes;
  p.off_slots = off;
  off += sizeof(int32_t) * static_cast<size_t>(tpc) * a.topk;
  p.off_active = off;
  off += sizeof(int32_t) * static_cast<size_t>(tpc);
  p.off_padpre = off;
  off += sizeof(int32_t) * (static_cast<size_t>(a.num_experts) + 1);
  p.smem = (off + 127) / 128 * 128;
  return p;
}

}  // namespace

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t stream) {
  const PermutePlan p = make_permute_plan(a, device_sm_count());
  cudaError_t st = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(p.smem));
  if (st != cudaSuccess) return st;
  st = launch_pdl(permute_kernel, dim3(static_cast<unsigned>(p.grid)), dim3(kPermuteThreads), p.smem, stream, a, p);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
