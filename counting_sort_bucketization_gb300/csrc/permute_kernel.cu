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
//    stores; gap rows are split evenly over CTAs by a prefix sum of gap sizes.
//
// Two kernels:
//  - permute_dyn_kernel (the default): a persistent grid of one wave (3 CTAs
//    per SM) whose TMA threads claim units -- pieces of token rows -- one at
//    a time from a counter in the workspace.  A measured trace of the
//    statically split kernel showed SMs with equal shares finishing as much
//    as 40 % apart, and a grid of 1.3 waves when rows are small; claiming
//    keeps every SM busy to the end, and cutting rows into pieces when a CTA
//    would see few rows keeps most units in the counter instead of in the
//    CTAs' rings.  A unit's slots and (with the row's first piece) its scale
//    factors come in by bulk copy on the same mbarrier as its bytes.
//  - permute_kernel: a static split of contiguous token blocks, used when a
//    row is wider than one 16 KiB slice or scale rows are not 16-byte sized.
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
// Ring of the dynamic kernel: up to MOE_PERMUTE_MAX_STAGES units, at most
// this many bytes.  Measured on GB300 at 3 CTAs per SM: 16 stages in 64 KB
// took decode's permute from 116.7 to 112.8 us (8 stages in 48 KB before);
// 24 stages in 96 KB left 2 CTAs per SM and took it to 144 us.
#ifndef MOE_PERMUTE_STAGE_BUDGET
#define MOE_PERMUTE_STAGE_BUDGET (64 * 1024)
#endif

constexpr int kPermuteThreads = 256;
constexpr int kPermuteWarps = kPermuteThreads / kWarpSize;
#ifndef MOE_PERMUTE_MAX_STAGES
#define MOE_PERMUTE_MAX_STAGES 16
#endif
constexpr int kMaxStages = MOE_PERMUTE_MAX_STAGES;
constexpr int kMaxChunkBytes = 16384;
constexpr int kStageBudgetBytes = MOE_PERMUTE_STAGE_BUDGET;  // shared-memory ring per CTA (dynamic kernel)
constexpr int kStaticMaxStages = 8;                          // the static kernel's ring: 8 stages in 48 KB
constexpr int kStaticStageBudget = 48 * 1024;
constexpr int kCtasPerSm = MOE_PERMUTE_CTAS_PER_SM;           // static kernel's grid target
constexpr int kMaxTokensPerCta = 512;
constexpr int kSfRegWords = 4;  // scale-factor words a lane keeps in registers
#ifndef MOE_PERMUTE_MIN_UNIT_BYTES
#define MOE_PERMUTE_MIN_UNIT_BYTES 3584
#endif
#ifndef MOE_PERMUTE_RANKS_MIN_UNIT_BYTES
#define MOE_PERMUTE_RANKS_MIN_UNIT_BYTES 7168
#endif
#ifndef MOE_PERMUTE_UNITS_PER_CTA
#define MOE_PERMUTE_UNITS_PER_CTA 48
#endif
// The dynamic kernel cuts rows into the fewest pieces that give each CTA at
// least kUnitsPerCta units, but no piece below kMinUnitBytes: a sweep of
// fixed piece sizes on GB300 put decode-sized batches (6-7 rows per CTA) at
// 0.88 of the copy peak with whole rows and 0.94 with 3.5 KB pieces, while
// pieces of 2 KB lost up to 12 % on the large batches.  The non-expand
// permute (one row per token and rank reached: ~5 of 8 slots hold a row on
// decode) wants larger pieces: 7 KB took its decode permute from 75.8 to
// 61.1 us, 3.5 KB pieces being no better for its larger batches.
#ifndef MOE_PERMUTE_L2_EVICT_FIRST
#define MOE_PERMUTE_L2_EVICT_FIRST 1
#endif
// CTAs of the dynamic kernel per SM (fewer if fewer fit).  Measured on
// GB300 with the same ring: 4 per SM beat 5 on every workload (decode
// permute 120.3 -> 116.5 us, skewed 324.5 -> 317.4, round-trip 1375.6 ->
// 1364.1) and 3 beat 4 by up to 1 % (prefill fp8 344.0 -> 340.5 us, decode
// unchanged); the L2 policy alone moved them by 0.2-0.4 %.
#ifndef MOE_PERMUTE_DYN_CTAS_PER_SM
#define MOE_PERMUTE_DYN_CTAS_PER_SM 3
#endif
#ifndef MOE_PERMUTE_DYN_MIN_BLOCKS
#define MOE_PERMUTE_DYN_MIN_BLOCKS MOE_PERMUTE_DYN_CTAS_PER_SM
#endif
constexpr int kMinUnitBytes = MOE_PERMUTE_MIN_UNIT_BYTES;
constexpr int kRanksMinUnitBytes = MOE_PERMUTE_RANKS_MIN_UNIT_BYTES;
constexpr int kUnitsPerCta = MOE_PERMUTE_UNITS_PER_CTA;
static_assert(kMinUnitBytes >= 16 && kMinUnitBytes % 16 == 0, "piece size");
static_assert(kRanksMinUnitBytes >= 16 && kRanksMinUnitBytes % 16 == 0, "piece size");

// Bulk store of receive rows, which nothing in the permute reads again: with
// an evict-first L2 policy their lines go first when L2 needs room.
__device__ __forceinline__ uint64_t store_policy() {
  return MOE_PERMUTE_L2_EVICT_FIRST ? ptx::l2_evict_first_policy() : 0;
}
__device__ __forceinline__ void store_rows(void* dst, const void* src, uint32_t bytes, uint64_t policy) {
  if (MOE_PERMUTE_L2_EVICT_FIRST)
    ptx::bulk_s2g_hint(dst, src, bytes, policy);
  else
    ptx::bulk_s2g(dst, src, bytes);
}

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

// gap_prefix computed by the helper warps alone (threads kWarpSize.., a named
// barrier instead of __syncthreads), so warp 0 never waits for it.
__device__ void gap_prefix_helpers(const int32_t* __restrict__ off, const int32_t* __restrict__ cnt, int E,
                                   int32_t* padpre, int* warp_tot) {
  constexpr int kHelp = kPermuteThreads - kWarpSize;
  const int h = threadIdx.x - kWarpSize;
  const int lane = h % kWarpSize, hw = h / kWarpSize;
  const int ipt = (E + kHelp - 1) / kHelp;
  const int e_lo = h * ipt;
  int mine = 0;
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) mine += __ldg(off + e + 1) - __ldg(off + e) - __ldg(cnt + e);
  }
  const int incl = warp_inclusive_scan(mine, lane);
  if (lane == kWarpSize - 1) warp_tot[hw] = incl;
  asm volatile("bar.sync 1, %0;" ::"r"(kHelp) : "memory");
  int run = incl - mine;
  for (int w = 0; w < hw; ++w) run += warp_tot[w];
  for (int j = 0; j < ipt; ++j) {
    const int e = e_lo + j;
    if (e < E) {
      padpre[e] = run;
      run += __ldg(off + e + 1) - __ldg(off + e) - __ldg(cnt + e);
    }
  }
  if (h == kHelp - 1) padpre[E] = run;
  asm volatile("bar.sync 1, %0;" ::"r"(kHelp) : "memory");
}

// This CTA's equal share of the gap rows (and their scale-factor rows) set to
// zero by the nhelp threads htid = 0..nhelp-1.
__device__ void zero_gap_share(const PermuteArgs& a, const int32_t* padpre_s, int E, int htid, int nhelp) {
  const int64_t total_pad = padpre_s[E];
  const int64_t G = gridDim.x;
  const int64_t p0 = total_pad * blockIdx.x / G, p1 = total_pad * (blockIdx.x + 1) / G;
  if (p0 >= p1) return;
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

// ------------------------------------------------------------ static split
struct PermutePlan {
  int chunk_bytes;     // bytes per bulk load (a row, or a 16 KiB slice of it)
  int nchunks;         // slices per row
  int stages;          // shared-memory ring depth
  int tokens_per_cta;
  int64_t grid;
  size_t off_slots, off_active, off_padpre, smem;
};

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

  // Slots of the CTA's tokens; kBatch independent loads per thread in flight.
  constexpr int kBatch = 8;
  for (int base = threadIdx.x; base < ntok * K; base += kBatch * kPermuteThreads) {
    int v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kPermuteThreads;
      v[u] = i < ntok * K ? __ldg(a.dst_slot + t0 * K + i) : -1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + u * kPermuteThreads;
      if (i >= ntok * K) break;
      int s = v[u];
      if (s >= a.capacity) {
        set_error(a.err, MOE_ERR_CAPACITY);
        s = -1;
      }
      slots_s[i] = s;
    }
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
    int issued = prologue;
    int u = 0;
    bool ok = true;
    const uint64_t policy = store_policy();
    for (; u < units; ++u) {
      const int s = u % S;
      if (!ptx::mbar_wait_parity_bounded(&full_bar[s], (u / S) & 1, a.wait_ns)) {
        ok = false;
        break;
      }
      const int tok = active_s[u / nch], c = u % nch;
      const uint32_t bytes = unit_bytes(c);
      const int32_t* sl = slots_s + tok * K;
      const uint8_t* src = ring + static_cast<size_t>(s) * chunk;
      for (int k = 0; k < K; ++k) {
        const int32_t slot = sl[k];
        if (slot >= 0) store_rows(a.recv_x + slot * rb + static_cast<int64_t>(c) * chunk, src, bytes, policy);
      }
      ptx::bulk_commit();
      if (u + S < units) {
        ptx::bulk_wait_read<0>();  // this stage's stores have read it
        issue(u + S);
        ++issued;
      }
    }
    if (!ok) {
      set_error(a.err, MOE_ERR_TIMEOUT);
      // Let the loads already issued land before the CTA's shared memory goes away.
      for (int v = u; v < issued; ++v)
        ptx::mbar_wait_parity_bounded(&full_bar[v % S], (v / S) & 1, a.wait_ns);
    }
    ptx::bulk_wait<0>();
    return;
  }

  // ---- helper warps: gap rows and scale-factor rows ------------------------
  const int htid = threadIdx.x - kWarpSize;
  const int nhelp = kPermuteThreads - kWarpSize;
  const int hwarp = warp - 1, nhwarps = kPermuteWarps - 1;
  if (a.zero_pad) zero_gap_share(a, padpre_s, E, htid, nhelp);
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
  p.stages = std::max(2, std::min(kStaticMaxStages, kStaticStageBudget / p.chunk_bytes));
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

// ------------------------------------------------------ dynamic (default)
// The unit of work is a piece of one token row (a "unit": the row cut into
// `pieces` of at most unit_bytes): a CTA holds several units in its ring
// for the bandwidth, and small units keep most of them in the shared
// counter, where whichever CTA is free first takes them.  With whole rows
// as units the first claims alone handed out ~3/4 of a 4096-token batch.
struct DynPlan {
  int row_bytes;     // <= kMaxChunkBytes, multiple of 16
  int unit_bytes;    // row bytes a unit moves (multiple of 16); the last piece of a row may be shorter
  int pieces;        // units per row
  int slot_win;      // bytes reserved per stage for the token's 16-byte-aligned slot window
  int sf_bytes;      // scale-factor row bytes (multiple of 16) or 0; moved with piece 0
  int stage_bytes;   // unit + slot window + scale row, rounded to 128
  int stages;
  int64_t grid;
  size_t off_padpre, smem;
};

__global__ void __launch_bounds__(kPermuteThreads, MOE_PERMUTE_DYN_MIN_BLOCKS)
    permute_dyn_kernel(const PermuteArgs a, const DynPlan p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ int warp_tot_s[kPermuteWarps];
  __shared__ int64_t stage_tok[kMaxStages];
  int32_t* padpre_s = reinterpret_cast<int32_t*>(smem + p.off_padpre);
  const int K = a.topk, E = a.num_experts;
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;

  if (warp != 0) {
    // Helper warps: this CTA's share of the gap rows, after the layout is done.
    ptx::grid_dependency_wait();
    if (__ldg(a.total_rows) > a.capacity || !a.zero_pad) return;
    gap_prefix_helpers(a.expert_offset, a.expert_count, E, padpre_s, warp_tot_s);
    zero_gap_share(a, padpre_s, E, threadIdx.x - kWarpSize, kPermuteThreads - kWarpSize);
    return;
  }
  if (lane != 0) return;

  // ---- the CTA's TMA thread ---------------------------------------------
  const int64_t N = a.num_tokens;
  const int64_t U = N * p.pieces;   // units: piece c of token t is unit t * pieces + c
  const int64_t rb = a.row_bytes, srb = a.sf_row_bytes;
  const int S = p.stages;
  const int64_t G = gridDim.x;
  unsigned* next_tok = a.work;
  unsigned* done_ctas = a.work + 1;
  const uintptr_t slots_lo = reinterpret_cast<uintptr_t>(a.dst_slot);
  const uintptr_t slots_hi = reinterpret_cast<uintptr_t>(a.dst_slot + N * K);
  // 16-byte-aligned window of dst_slot holding token t's K slots; when it
  // would reach outside the array the slots are read directly instead.
  auto window_of = [&](int64_t t, uintptr_t& w0, uintptr_t& w1, uintptr_t& first) -> bool {
    first = reinterpret_cast<uintptr_t>(a.dst_slot + t * K);
    w0 = first & ~uintptr_t(15);
    w1 = (first + 4u * static_cast<unsigned>(K) + 15) & ~uintptr_t(15);
    return w0 >= slots_lo && w1 <= slots_hi;
  };
  for (int s = 0; s < S; ++s) ptx::mbar_init(&full_bar[s], 1);
  ptx::fence_mbar_init();

  // Unit u: token u / pieces, bytes [off, off + len) of its row; piece 0
  // also carries the token's scale row.
  auto piece_of = [&](int64_t u, int64_t& t, int64_t& off, uint32_t& len, bool& with_sf) {
    t = u / p.pieces;
    const int c = static_cast<int>(u - t * p.pieces);
    off = static_cast<int64_t>(c) * p.unit_bytes;
    len = static_cast<uint32_t>(min64(p.unit_bytes, rb - off));
    with_sf = p.sf_bytes != 0 && c == 0;
  };
  // The first S units of every CTA are fixed (blockIdx.x + i*G): their rows
  // and scale rows do not depend on the layout, so they are requested before
  // waiting for the previous kernel.  Each stage's phase completes only after
  // the post-wait arrival, which also brings the slot window.
  int npre = 0;
  for (; npre < S; ++npre) {
    const int64_t u = blockIdx.x + npre * G;
    if (u >= U) break;
    int64_t t, off;
    uint32_t len;
    bool with_sf;
    piece_of(u, t, off, len, with_sf);
    uint8_t* st = smem + static_cast<size_t>(npre) * p.stage_bytes;
    stage_tok[npre] = u;
    // a.extra_tx is 0 except under the timeout test hook: bytes no copy delivers.
    ptx::mbar_expect_tx(&full_bar[npre], len + (with_sf ? static_cast<uint32_t>(p.sf_bytes) : 0u) +
                                             (npre == 0 ? a.extra_tx : 0u));
    ptx::bulk_g2s(st, a.x + t * rb + off, len, &full_bar[npre]);
    if (with_sf)
      ptx::bulk_g2s(st + p.unit_bytes + p.slot_win, a.sf + t * srb, static_cast<uint32_t>(p.sf_bytes),
                    &full_bar[npre]);
  }
  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  const bool cap_ok = __ldg(a.total_rows) <= a.capacity;   // uniform over the grid
  if (!cap_ok) {
    if (blockIdx.x == 0) set_error(a.err, MOE_ERR_CAPACITY);
    for (int i = 0; i < npre; ++i) ptx::mbar_arrive(&full_bar[i]);
    for (int i = 0; i < npre; ++i) ptx::mbar_wait_parity_bounded(&full_bar[i], 0, a.wait_ns);
    return;   // no CTA touches the token counter
  }
  for (int i = 0; i < npre; ++i) {
    uintptr_t w0, w1, first;
    if (window_of(stage_tok[i] / p.pieces, w0, w1, first)) {
      ptx::mbar_arrive_expect_tx(&full_bar[i], static_cast<uint32_t>(w1 - w0));
      ptx::bulk_g2s(smem + static_cast<size_t>(i) * p.stage_bytes + p.unit_bytes, reinterpret_cast<const void*>(w0),
                    static_cast<uint32_t>(w1 - w0), &full_bar[i]);
    } else {
      ptx::mbar_arrive(&full_bar[i]);
    }
  }

  // Later units are claimed from the counter (claim c is unit G*S + c),
  // two claims ahead of use so the atomic's latency is hidden.
  const int64_t claimed_base = G * S;
  int64_t claim0 = claimed_base + atomicAdd(next_tok, 1u), claim1 = claimed_base + atomicAdd(next_tok, 1u);
  bool exhausted = npre < S;
  int64_t issued = npre;
  auto issue = [&]() {
    const int64_t u = claim0;
    claim0 = claim1;
    if (u >= U) {
      exhausted = true;
      return;
    }
    claim1 = claimed_base + atomicAdd(next_tok, 1u);
    int64_t t, off;
    uint32_t len;
    bool with_sf;
    piece_of(u, t, off, len, with_sf);
    const int s = static_cast<int>(issued % S);
    uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
    stage_tok[s] = u;
    uintptr_t w0, w1, first;
    const bool window = window_of(t, w0, w1, first);
    const uint32_t tx = len + (window ? static_cast<uint32_t>(w1 - w0) : 0u) +
                        (with_sf ? static_cast<uint32_t>(p.sf_bytes) : 0u);
    ptx::mbar_arrive_expect_tx(&full_bar[s], tx);
    ptx::bulk_g2s(st, a.x + t * rb + off, len, &full_bar[s]);
    if (window)
      ptx::bulk_g2s(st + p.unit_bytes, reinterpret_cast<const void*>(w0), static_cast<uint32_t>(w1 - w0),
                    &full_bar[s]);
    if (with_sf)
      ptx::bulk_g2s(st + p.unit_bytes + p.slot_win, a.sf + t * srb, static_cast<uint32_t>(p.sf_bytes), &full_bar[s]);
    ++issued;
  };
  int64_t j = 0;
  bool ok = true;
  const uint64_t policy = store_policy();
  for (; j < issued; ++j) {
    const int s = static_cast<int>(j % S);
    if (!ptx::mbar_wait_parity_bounded(&full_bar[s], static_cast<uint32_t>((j / S) & 1), a.wait_ns)) {
      ok = false;
      break;
    }
    int64_t t, off;
    uint32_t len;
    bool with_sf;
    piece_of(stage_tok[s], t, off, len, with_sf);
    const uint8_t* st = smem + static_cast<size_t>(s) * p.stage_bytes;
    uintptr_t w0, w1, first;
    const bool window = window_of(t, w0, w1, first);
    const int32_t* sl = window ? reinterpret_cast<const int32_t*>(st + p.unit_bytes + (first - w0)) : nullptr;
    for (int k = 0; k < K; ++k) {
      const int32_t slot = window ? sl[k] : __ldg(a.dst_slot + t * K + k);
      if (slot < 0) continue;
      if (slot >= a.capacity) {
        if (off == 0) set_error(a.err, MOE_ERR_CAPACITY);
        continue;
      }
      store_rows(a.recv_x + slot * rb + off, st, len, policy);
      if (with_sf)
        store_rows(a.recv_sf + slot * srb, st + p.unit_bytes + p.slot_win, static_cast<uint32_t>(srb), policy);
    }
    ptx::bulk_commit();
    if (!exhausted) {
      ptx::bulk_wait_read<0>();  // this stage's stores have read it
      issue();
    }
  }
  if (!ok) {
    set_error(a.err, MOE_ERR_TIMEOUT);
    for (int64_t v = j; v < issued; ++v)
      ptx::mbar_wait_parity_bounded(&full_bar[v % S], static_cast<uint32_t>((v / S) & 1), a.wait_ns);
  }
  ptx::bulk_wait<0>();
  // The fence orders this CTA's claims before its arrival below; the last
  // CTA to arrive resets both counters for the next launch on the workspace.
  __threadfence();
  if (atomicAdd(done_ctas, 1u) == gridDim.x - 1) {
    atomicExch(next_tok, 0u);
    atomicExch(done_ctas, 0u);
  }
}

int max_pieces(const PermuteArgs& a) {
  const int min_unit = a.non_expand ? kRanksMinUnitBytes : kMinUnitBytes;
  return static_cast<int>(max64(1, ceil_div64(a.row_bytes, min_unit)));
}

bool dyn_applicable(const PermuteArgs& a) {
  if (a.row_bytes > kMaxChunkBytes || a.work == nullptr) return false;
  // Unit indices (and the claims past them) must fit the 32-bit counter.
  if (a.num_tokens * max_pieces(a) >= (int64_t{1} << 31)) return false;
  if (a.sf != nullptr) {
    if (a.sf_row_bytes % 16 != 0 || a.sf_row_bytes > 4096) return false;
    if (reinterpret_cast<uintptr_t>(a.sf) % 16 != 0 || reinterpret_cast<uintptr_t>(a.recv_sf) % 16 != 0) return false;
  }
  return true;
}

// Plan for rows cut into (about) `pieces` equal 16-byte-multiple pieces; the
// piece count is recomputed from the rounded size, so the last piece is
// never empty.
DynPlan make_dyn_plan(const PermuteArgs& a, int pieces) {
  DynPlan p{};
  p.row_bytes = static_cast<int>(a.row_bytes);
  p.unit_bytes = static_cast<int>(ceil_div64(ceil_div64(a.row_bytes, max64(1, pieces)), 16) * 16);
  p.pieces = static_cast<int>(ceil_div64(a.row_bytes, p.unit_bytes));
  p.slot_win = static_cast<int>((4 * a.topk + 32 + 15) / 16 * 16);
  p.sf_bytes = a.sf != nullptr ? static_cast<int>(a.sf_row_bytes) : 0;
  p.stage_bytes = (p.unit_bytes + p.slot_win + p.sf_bytes + 127) / 128 * 128;
  p.stages = std::max(2, std::min(kMaxStages, kStageBudgetBytes / p.stage_bytes));
  size_t off = static_cast<size_t>(p.stages) * p.stage_bytes;
  p.off_padpre = off;
  off += sizeof(int32_t) * (static_cast<size_t>(a.num_experts) + 1);
  p.smem = (off + 127) / 128 * 128;
  return p;
}

// CTAs of the dynamic kernel resident per SM at this shared-memory size (cached).
int dyn_ctas_per_sm(size_t smem) {
  const int occ = cached_occupancy(permute_dyn_kernel, kPermuteThreads, smem);
  return occ < 1 ? 1 : occ;
}

}  // namespace

cudaError_t launch_permute(const PermuteArgs& args, cudaStream_t stream) {
  PermuteArgs a = args;
  const WaitConfig wc = wait_config();
  a.wait_ns = wc.limit_ns;
  a.extra_tx = wc.extra_tx;
  if (dyn_applicable(a)) {
    DynPlan p = make_dyn_plan(a, 1);
    auto ctas_per_sm = [](size_t smem) {
      const int occ = dyn_ctas_per_sm(smem);
      return MOE_PERMUTE_DYN_CTAS_PER_SM > 0 && MOE_PERMUTE_DYN_CTAS_PER_SM < occ ? MOE_PERMUTE_DYN_CTAS_PER_SM : occ;
    };
    int64_t resident = static_cast<int64_t>(ctas_per_sm(p.smem)) * device_sm_count();
    const int64_t want = ceil_div64(kUnitsPerCta * resident, max64(1, a.num_tokens));
    const int pieces = static_cast<int>(min64(want, max_pieces(a)));
    if (pieces > 1) {
      p = make_dyn_plan(a, pieces);
      resident = static_cast<int64_t>(ctas_per_sm(p.smem)) * device_sm_count();
    }
    cudaError_t st = ensure_smem_limit(permute_dyn_kernel, p.smem);
    if (st != cudaSuccess) return st;
    p.grid = max64(1, min64(resident, a.num_tokens * p.pieces));
    st = launch_pdl(permute_dyn_kernel, dim3(static_cast<unsigned>(p.grid)), dim3(kPermuteThreads), p.smem, stream,
                    a, p);
    if (st != cudaSuccess) return st;
    count_launch();
    return cudaSuccess;
  }
  const PermutePlan p = make_permute_plan(a, device_sm_count());
  cudaError_t st = ensure_smem_limit(permute_kernel, p.smem);
  if (st != cudaSuccess) return st;
  st = launch_pdl(permute_kernel, dim3(static_cast<unsigned>(p.grid)), dim3(kPermuteThreads), p.smem, stream, a, p);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
