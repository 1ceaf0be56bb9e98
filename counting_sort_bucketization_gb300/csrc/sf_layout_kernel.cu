// sf_layout_kernel.cu -- the scale factors of a receive buffer in
// column-major, TMA-aligned form.
//
// Method: page "00 DeepEP Engram Architecture Deep-Dive", §1.1-§1.2, names
// the fetch option use_tma_aligned_col_major_sf and does not define it.  The
// reading taken: the [rows, C] matrix of 4-byte scale words is stored column
// after column, column j at out + j*ld, with ld a multiple of 4 words so that
// every column starts on a 16-byte boundary (a TMA global stride must be a
// multiple of 16 bytes).  Rows move as in the dispatch permute of page
// "07 DeepEP Counting Sort / Bucketization" (§6.4, §8.2), and the alignment
// gap rows are zero (§7.3).
//
// Design: a gather.  A CTA takes tiles of 128 receive rows; the inverse map
// (src_idx, or rank_src) names each row's token.  Each warp reads whole
// token scale rows (lanes along the row, coalesced) into a shared-memory
// tile, and the tile goes out as 512-byte runs of each column, so every
// global store covers full 32-byte sectors in address order.  A scatter from
// the token side would write 4 scattered bytes per column per copy.
//
// The shared tile is swizzled so that both phases are free of bank
// conflicts: word (row i, column j) sits in column j's 128-word line at
// 4-row group (i/4) ^ ((j/4) % 8), position (i ^ j) % 4 inside the group.  A
// warp writing one row's 32 columns then touches 32 different banks, and a
// lane reading one column's 4-row group finds it contiguous (one 16-byte
// load, components permuted by j % 4).
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kSfThreads = 256;
constexpr int kSfWarps = kSfThreads / kWarpSize;
constexpr int kSfTileRows = 128;                          // receive rows per tile
constexpr int kSfPassCols = 64;                           // columns per pass through the tile
constexpr int kSfRowsPerWarp = kSfTileRows / kSfWarps;   // 16
constexpr int kSfBatch = 8;                               // rows whose loads a lane keeps in flight
constexpr int kSfColsPerLane = kSfPassCols / kWarpSize;  // 2
constexpr int32_t kPastRows = -2;                         // src_s marker: row not written

static_assert(kSfTileRows == 4 * kWarpSize, "one 4-row group per lane in the store phase");
static_assert(kSfRowsPerWarp % kSfBatch == 0, "whole batches per warp");

__device__ __forceinline__ int tile_word(int i, int j) {
  return j * kSfTileRows + (((i >> 2) ^ ((j >> 2) & 7)) << 2) + ((i ^ j) & 3);
}

__global__ void __launch_bounds__(kSfThreads) sf_col_major_kernel(const SfColMajorArgs a) {
  extern __shared__ __align__(16) uint32_t tile[];   // [pass_cols][kSfTileRows], swizzled
  __shared__ __align__(16) int32_t src_s[kSfTileRows];
  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  const int64_t C = a.cols;

  ptx::grid_dependency_wait();
  ptx::grid_dependency_launch_dependents();
  const int64_t rows = __ldg(a.total_rows);
  if (rows > a.capacity || rows < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, MOE_ERR_CAPACITY);
    return;
  }
  const int64_t tiles = ceil_div64(rows, kSfTileRows);
  for (int64_t tile_i = blockIdx.x; tile_i < tiles; tile_i += gridDim.x) {
    const int64_t r0 = tile_i * kSfTileRows;
    __syncthreads();   // the previous tile's stores have read src_s and the tile
    if (threadIdx.x < kSfTileRows) {
      const int64_t r = r0 + threadIdx.x;
      int32_t t = kPastRows;
      if (r < rows) {
        t = __ldg(a.src + r);
        if (t < -1 || t >= a.num_tokens) {
          set_error(a.err, MOE_ERR_INVALID_ARG);
          t = kPastRows;
        } else if (t == -1 && !a.zero_pad) {
          t = kPastRows;
        }
      }
      src_s[threadIdx.x] = t;
    }
    __syncthreads();

    for (int64_t c0 = 0; c0 < C; c0 += kSfPassCols) {
      const int nc = static_cast<int>(min64(kSfPassCols, C - c0));
      if (c0 > 0) __syncthreads();   // the previous pass's stores are done with the tile
      // Gather: warp w fills rows [16w, 16w + 16); lane l holds columns l, l + 32.
#pragma unroll
      for (int b = 0; b < kSfRowsPerWarp; b += kSfBatch) {
        uint32_t v[kSfBatch][kSfColsPerLane];
#pragma unroll
        for (int u = 0; u < kSfBatch; ++u) {
          const int32_t t = src_s[warp * kSfRowsPerWarp + b + u];
          const uint32_t* row = a.sf + static_cast<int64_t>(t >= 0 ? t : 0) * C + c0;
#pragma unroll
          for (int h = 0; h < kSfColsPerLane; ++h) {
            const int j = lane + h * kWarpSize;
            v[u][h] = (t >= 0 && j < nc) ? __ldg(row + j) : 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < kSfBatch; ++u) {
          const int i = warp * kSfRowsPerWarp + b + u;
#pragma unroll
          for (int h = 0; h < kSfColsPerLane; ++h) {
            const int j = lane + h * kWarpSize;
            if (j < nc) tile[tile_word(i, j)] = v[u][h];
          }
        }
      }
      __syncthreads();
      // Store: warp w writes columns w, w + 8, ...; lane l writes rows 4l .. 4l + 3.
      const int4 flags = *reinterpret_cast<const int4*>(&src_s[4 * lane]);
      const bool w0 = flags.x != kPastRows, w1 = flags.y != kPastRows;
      const bool w2 = flags.z != kPastRows, w3 = flags.w != kPastRows;
      for (int j = warp; j < nc; j += kSfWarps) {
        const uint4 g = *reinterpret_cast<const uint4*>(&tile[j * kSfTileRows + ((lane ^ ((j >> 2) & 7)) << 2)]);
        uint32_t o0 = g.x, o1 = g.y, o2 = g.z, o3 = g.w;   // row 4l + m sits in component m ^ (j % 4)
        if (j & 1) {
          const uint32_t s0 = o0, s2 = o2;
          o0 = o1; o1 = s0; o2 = o3; o3 = s2;
        }
        if (j & 2) {
          const uint32_t s0 = o0, s1 = o1;
          o0 = o2; o1 = o3; o2 = s0; o3 = s1;
        }
        uint32_t* dst = a.out + (c0 + j) * a.ld + r0 + 4 * lane;
        if (w0 && w1 && w2 && w3) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(o0, o1, o2, o3);
        } else {
          if (w0) dst[0] = o0;
          if (w1) dst[1] = o1;
          if (w2) dst[2] = o2;
          if (w3) dst[3] = o3;
        }
      }
    }
  }
}

size_t sf_smem_bytes(int64_t cols) {
  return static_cast<size_t>(min64(cols, kSfPassCols)) * kSfTileRows * sizeof(uint32_t);
}

// Resident CTAs per SM at a given dynamic shared-memory size (cached; at most
// kSfPassCols different sizes exist).
int sf_ctas_per_sm(size_t smem) {
  static std::mutex mu;
  static int cached[kSfPassCols + 1][8] = {};   // [columns in a pass][device]
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8) return 1;
  const size_t cols = smem / (kSfTileRows * sizeof(uint32_t));
  std::lock_guard<std::mutex> lock(mu);
  int& occ = cached[cols][dev];
  if (occ == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, sf_col_major_kernel, kSfThreads, smem) != cudaSuccess ||
        v < 1)
      v = 1;
    occ = v;
  }
  return occ;
}

}  // namespace

cudaError_t launch_sf_col_major(const SfColMajorArgs& a, cudaStream_t stream) {
  const size_t smem = sf_smem_bytes(a.cols);
  const int64_t tiles_max = max64(1, ceil_div64(a.capacity, kSfTileRows));
  const int64_t resident = static_cast<int64_t>(sf_ctas_per_sm(smem)) * device_sm_count();
  const int64_t grid = max64(1, min64(tiles_max, resident));
  const cudaError_t st = launch_pdl(sf_col_major_kernel, dim3(static_cast<unsigned>(grid)), dim3(kSfThreads), smem,
                                    stream, a);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
