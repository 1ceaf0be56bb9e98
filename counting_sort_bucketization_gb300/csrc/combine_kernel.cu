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
// HBM-bound: each thread owns 16-byte column vectors of the row and issues
// the loads of up to 8 expert rows before any arithmetic, so 8 x 16 B per
// thread are in flight; slots and weights of the CTA's token block are staged
// in shared memory once.
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

// Resident CTAs per SM at the largest shared-memory size a launch uses (cached per device).
int combine_ctas_per_sm() {
  const size_t smem = (sizeof(int32_t) + sizeof(float)) * kMaxTokensPerCta * MOE_MAX_TOPK;
  const int occ = cached_occupancy(combine_kernel, kCombineThreads, smem);
  return occ < 1 ? 1 : occ;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
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
