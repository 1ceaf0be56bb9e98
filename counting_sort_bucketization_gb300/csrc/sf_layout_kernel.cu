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
// When a scale row is a whole number of 16-byte chunks (C % 4 == 0) each
// half-warp loads one row with one 16-byte load per lane; otherwise lanes
// load single words.  The map entries of a CTA's next tile are requested
// before the current tile's rows, so one of the tile's two dependent global
// round trips overlaps the previous tile.
//
// Shared tile: column j of the tile is a line of 129 words starting at word
// 129*j + j/32, row i at offset i.  With that pitch every phase is free of
// bank conflicts: 32 lanes storing 32 columns of one row; the 16-byte loads'
// lanes storing word m of 4-word chunks of rows i and i + 2; and 32 lanes
// reading 32 consecutive rows of one column, which they then store as one
// 128-byte run of the output column.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kSfThreads = 256;
constexpr int kSfWarps = kSfThreads / kWarpSize;
constexpr int kSfTileRows = 128;                          // receive rows per tile
constexpr int kSfLine = kSfTileRows + 1;                  // words per column line of the tile
constexpr int kSfPassCols = 64;                           // columns per pass through the tile
constexpr int kSfRowsPerWarp = kSfTileRows / kSfWarps;   // 16
constexpr int kSfBatch = 8;                               // rows whose word loads a lane keeps in flight
constexpr int kSfColsPerLane = kSfPassCols / kWarpSize;  // 2
constexpr int kSfChunksPerRow = kSfPassCols / 4;          // 16-byte chunks of a pass's row: one half-warp
constexpr int kSfRunsPerColumn = kSfTileRows / kWarpSize; // 128-byte output runs per column of a tile
constexpr int32_t kPastRows = -2;                         // src_s marker: row not written

static_assert(kSfRowsPerWarp % kSfBatch == 0, "whole batches per warp");
static_assert(2 * kSfChunksPerRow == kWarpSize, "a warp's 16-byte loads cover two rows of a pass");
static_assert(kSfRowsPerWarp == 16, "the 16-byte gather walks rows in the order of vec_row");

__host__ __device__ __forceinline__ int line_start(int j) { return j * kSfLine + (j >> 5); }

// Row (within a warp's 16) that half-warp `half` loads in step p of the
// 16-byte gather: steps pair rows {0,2}, {1,3}, {4,6}, {5,7}, ...
__device__ __forceinline__ int vec_row(int p, int half) { return (((p >> 1) << 2) | (p & 1)) + 2 * half; }

// Map entry of receive row r as the tile uses it: a token, -1 (gap row to
// zero), or kPastRows (not written: past the rows, a gap row without
// zero_pad, or an entry out of range, which is reported).
__device__ __forceinline__ int32_t row_source(const SfColMajorArgs& a, int32_t t, int64_t r, int64_t rows) {
  if (r >= rows) return kPastRows;
  if (t < -1 || t >= a.num_tokens) {
    set_error(a.err, MOE_ERR_INVALID_ARG);
    return kPastRows;
  }
  return (t == -1 && !a.zero_pad) ? kPastRows : t;
}

template <bool kVec>
__global__ void __launch_bounds__(kSfThreads) sf_col_major_kernel(const SfColMajorArgs a) {
  extern __shared__ __align__(16) uint32_t tile[];   // pass_cols lines of kSfLine words
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
  // Threads below kSfTileRows carry the map entry of their row of the next tile.
  int32_t next_src = -1;
  if (threadIdx.x < kSfTileRows && static_cast<int64_t>(blockIdx.x) * kSfTileRows + threadIdx.x < rows)
    next_src = __ldg(a.src + static_cast<int64_t>(blockIdx.x) * kSfTileRows + threadIdx.x);
  for (int64_t tile_i = blockIdx.x; tile_i < tiles; tile_i += gridDim.x) {
    const int64_t r0 = tile_i * kSfTileRows;
    __syncthreads();   // the previous tile's stores have read src_s and the tile
    if (threadIdx.x < kSfTileRows) {
      src_s[threadIdx.x] = row_source(a, next_src, r0 + threadIdx.x, rows);
      const int64_t rn = r0 + static_cast<int64_t>(gridDim.x) * kSfTileRows + threadIdx.x;
      if (rn < rows) next_src = __ldg(a.src + rn);
    }
    __syncthreads();
    // Rows lane l stores: l + 32c for c < kSfRunsPerColumn.
    bool keep[kSfRunsPerColumn];
#pragma unroll
    for (int c = 0; c < kSfRunsPerColumn; ++c) keep[c] = src_s[lane + kWarpSize * c] != kPastRows;

    for (int64_t c0 = 0; c0 < C; c0 += kSfPassCols) {
      const int nc = static_cast<int>(min64(kSfPassCols, C - c0));
      if (c0 > 0) __syncthreads();   // the previous pass's stores are done with the tile
      if constexpr (kVec) {
        // Gather: warp w fills rows [16w, 16w + 16), two rows per load;
        // lane l holds chunk l % 16 (columns 4q .. 4q + 3) of its half's row.
        const int q = lane % kSfChunksPerRow;
        const int half = lane / kSfChunksPerRow;
        constexpr int kSteps = kSfRowsPerWarp / 2;
        uint4 v[kSteps];
#pragma unroll
        for (int p = 0; p < kSteps; ++p) {
          const int32_t t = src_s[warp * kSfRowsPerWarp + vec_row(p, half)];
          const uint4* row = reinterpret_cast<const uint4*>(a.sf + static_cast<int64_t>(t >= 0 ? t : 0) * C + c0);
          v[p] = (t >= 0 && 4 * q < nc) ? __ldg(row + q) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (4 * q < nc) {
          uint32_t* base = tile + line_start(4 * q) + warp * kSfRowsPerWarp;
#pragma unroll
          for (int p = 0; p < kSteps; ++p) {
            const int i = vec_row(p, half);
            base[i] = v[p].x;
            base[kSfLine + i] = v[p].y;
            base[2 * kSfLine + i] = v[p].z;
            base[3 * kSfLine + i] = v[p].w;
          }
        }
      } else {
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
          for (int h = 0; h < kSfColsPerLane; ++h) {
            const int j = lane + h * kWarpSize;
            if (j < nc) {
              uint32_t* base = tile + line_start(j) + warp * kSfRowsPerWarp + b;
#pragma unroll
              for (int u = 0; u < kSfBatch; ++u) base[u] = v[u][h];
            }
          }
        }
      }
      __syncthreads();
      // Store: warp w writes columns w, w + 8, ...; each lane one row of each
      // 32-row run, so a warp's store is 128 contiguous bytes of the column.
      for (int j = warp; j < nc; j += kSfWarps) {
        const uint32_t* line = tile + line_start(j) + lane;
        uint32_t* dst = a.out + (c0 + j) * a.ld + r0 + lane;
#pragma unroll
        for (int c = 0; c < kSfRunsPerColumn; ++c)
          if (keep[c]) dst[kWarpSize * c] = line[kWarpSize * c];
      }
    }
  }
}

size_t sf_smem_bytes(int64_t cols) {
  const int64_t pass = min64(cols, kSfPassCols);
  return static_cast<size_t>(line_start(static_cast<int>(pass))) * sizeof(uint32_t);
}

// Resident CTAs per SM of one kernel variant at a given dynamic shared-memory
// size (cached per device).
int sf_ctas_per_sm(bool vec, size_t smem) {
  const int occ = vec ? cached_occupancy(sf_col_major_kernel<true>, kSfThreads, smem)
                      : cached_occupancy(sf_col_major_kernel<false>, kSfThreads, smem);
  return occ < 1 ? 1 : occ;
}

}  // namespace

cudaError_t launch_sf_col_major(const SfColMajorArgs& a, cudaStream_t stream) {
  // 16-byte loads need every row (and so every pass of kSfPassCols words) to start 16-byte aligned.
  const bool vec = a.cols % 4 == 0 && reinterpret_cast<uintptr_t>(a.sf) % 16 == 0;
  const size_t smem = sf_smem_bytes(a.cols);
  const int64_t tiles_max = max64(1, ceil_div64(a.capacity, kSfTileRows));
  const int64_t resident = static_cast<int64_t>(sf_ctas_per_sm(vec, smem)) * device_sm_count();
  const int64_t grid = max64(1, min64(tiles_max, resident));
  const dim3 g(static_cast<unsigned>(grid)), b(kSfThreads);
  const cudaError_t st = vec ? launch_pdl(sf_col_major_kernel<true>, g, b, smem, stream, a)
                             : launch_pdl(sf_col_major_kernel<false>, g, b, smem, stream, a);
  if (st != cudaSuccess) return st;
  count_launch();
  return cudaSuccess;
}

}  // namespace moe
