/*
 * oracle.c -- CPU oracle for the MoE dispatch layout (counting sort /
 * bucketization) and its inverse combine.
 *
 * TEST INFRASTRUCTURE.  Plain, slow, single-threaded C.  Only the tests, the
 * smoke check and the CPU-baseline legs of the benchmark load it.  It shares
 * no code, header or constant with the CUDA library, and the library never
 * calls it.  Every step follows the page
 *   "07 DeepEP Counting Sort / Bucketization 深度校验：博客第一性原理 vs 源码实现"
 *   (DeepEP v2 source notes), cited below as [CS] with its section numbers.
 * The column-major scale-factor layout follows an option named on the page
 * "00 DeepEP Engram Architecture Deep-Dive", cited as [EA].
 *
 * Notation: N tokens, K top-k slots per token, E experts, R logical ranks,
 * L = E / R experts per rank, A the expert alignment.  topk_idx[t*K + k] is
 * the expert chosen by slot k of token t; a negative entry is masked.
 *
 * Readings taken where the pages leave a step open:
 *  - order inside an expert segment is (token, k) ascending: the pages hand
 *    out slots with atomics ([CS] §6.2, §6.4), so any order is valid for them;
 *    this oracle takes the one a sequential cursor gives;
 *  - alignment is applied to each expert's count before the exclusive sum
 *    ([CS] §7.2), so every segment starts on a multiple of A;
 *  - one global buffer: rank r's experts are e in [r*L, (r+1)*L), laid out
 *    rank after rank; offsets are one exclusive sum over all E experts;
 *  - an id >= E is reported as an error and the pair is dropped;
 *  - combine: fp32 accumulator starting at 0, k ascending, one fused
 *    multiply-add per term (fmaf), one round-to-nearest-even to bf16 at the
 *    end; masked slots are skipped.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_EXPERT_ID 2
#define ORACLE_CAPACITY 3

/* [CS] §7.2: align(x, a) rounds x up to the next multiple of a. */
static int64_t align_up(int64_t x, int64_t a) { return ((x + a - 1) / a) * a; }

/*
 * oracle_layout -- count, prefix sums and the expert-major slot maps.
 *
 *  [CS] §4.2   expert_count[e] = number of (t,k) with topk_idx == e;
 *              rank_count[r]   = number of tokens with at least one valid id
 *                                in rank r (r = e / L), each token once.
 *  [CS] §7.2   aligned count of expert e = align(expert_count[e], A).
 *  [CS] §5.2/§5.5  expert_offset = exclusive sum of the aligned counts
 *              ([E+1] entries, the last one is the row total);
 *              rank_psum = inclusive sum of rank_count.
 *  [CS] §6.4   the exclusive sum is then used as a per-expert cursor: every
 *              valid pair, visited in (t,k) order, takes the cursor's value
 *              as its slot and advances it.
 *  dst_slot[t*K+k] = slot (or -1 if masked / dropped);
 *  src_idx[slot] = t; rows in the alignment gap keep src_idx = -1.
 *
 * Returns ORACLE_CAPACITY (and leaves dst_slot/src_idx untouched) when the
 * row total exceeds capacity_rows; ORACLE_BAD_EXPERT_ID when an id >= E was
 * seen (all outputs are still written, the bad pairs being dropped).
 */
int oracle_layout(int64_t N, int32_t K, int32_t E, int32_t R, int32_t A,
                  const int64_t *topk_idx, int32_t *expert_count,
                  int32_t *rank_count, int32_t *expert_offset,
                  int32_t *rank_psum, int32_t *dst_slot, int32_t *src_idx,
                  int64_t capacity_rows, int64_t *total_rows) {
  if (N < 0 || K < 1 || E < 1 || R < 1 || A < 1 || E % R != 0)
    return ORACLE_BAD_ARG;
  const int32_t L = E / R;
  int status = ORACLE_OK;

  /* Count ([CS] §4.2). last_token[r] remembers the last token that was
     already counted for rank r, so a token adds at most one to each rank. */
  int64_t *last_token = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
  if (!last_token) return ORACLE_BAD_ARG;
  for (int32_t r = 0; r < R; ++r) last_token[r] = -1;
  for (int32_t e = 0; e < E; ++e) expert_count[e] = 0;
  for (int32_t r = 0; r < R; ++r) rank_count[r] = 0;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0) continue;
      if (e >= E) { status = ORACLE_BAD_EXPERT_ID; continue; }
      expert_count[e] += 1;
      int32_t r = (int32_t)(e / L);
      if (last_token[r] != t) {
        last_token[r] = t;
        rank_count[r] += 1;
      }
    }
  }
  free(last_token);

  /* Align, then exclusive sum over experts ([CS] §7.2, §5.5). */
  int64_t run = 0;
  expert_offset[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    run += align_up(expert_count[e], A);
    expert_offset[e + 1] = (int32_t)run;
  }
  /* Inclusive sum over ranks ([CS] §5.5). */
  int64_t rrun = 0;
  for (int32_t r = 0; r < R; ++r) {
    rrun += rank_count[r];
    rank_psum[r] = (int32_t)rrun;
  }
  *total_rows = run;
  if (run > capacity_rows) return ORACLE_CAPACITY;

  /* Scatter with the exclusive sum as cursor ([CS] §6.4). */
  int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  if (!cursor) return ORACLE_BAD_ARG;
  for (int32_t e = 0; e < E; ++e) cursor[e] = expert_offset[e];
  for (int64_t i = 0; i < run; ++i) src_idx[i] = -1;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0 || e >= E) {
        dst_slot[t * K + k] = -1;
        continue;
      }
      int32_t s = cursor[e]++;
      dst_slot[t * K + k] = s;
      src_idx[s] = (int32_t)t;
    }
  }
  free(cursor);
  return status;
}

/*
 * oracle_rank_layout -- the non-expand (rank-contiguous) slot map
 * ([CS] §6.2 "Scatter 1", §8.1-§8.2).
 *
 * Each token is copied once per logical rank it reaches (deduplicated, as
 * in the count of [CS] §4.2).  Rank r's block of rows starts at the
 * exclusive sum of rank_count over earlier ranks; inside it tokens are in
 * ascending order (the page hands out these slots with an atomic counter,
 * so any order is valid for it).  Of the token's top-k slots that reach
 * rank r, the highest k (the page's "master lane", the highest lane of the
 * group) gets the row; the others, and masked slots, get -1.
 *   rank_slot[t*K+k]: row in the rank-contiguous buffer or -1;
 *   rank_src[row]:    token of each row ([rows], rows = sum of rank_count).
 * Ids >= E are dropped as in oracle_layout.  Returns ORACLE_CAPACITY if the
 * rows exceed capacity_rows (maps untouched), ORACLE_BAD_EXPERT_ID if a bad
 * id was seen.
 */
int oracle_rank_layout(int64_t N, int32_t K, int32_t E, int32_t R,
                       const int64_t *topk_idx, int32_t *rank_slot,
                       int32_t *rank_src, int64_t capacity_rows,
                       int64_t *total_rows) {
  if (N < 0 || K < 1 || E < 1 || R < 1 || E % R != 0) return ORACLE_BAD_ARG;
  const int32_t L = E / R;
  int status = ORACLE_OK;
  /* Rank counts, one per token per rank ([CS] §4.2). */
  int64_t *count = (int64_t *)calloc((size_t)R, sizeof(int64_t));
  int64_t *last_token = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
  if (!count || !last_token) return ORACLE_BAD_ARG;
  for (int32_t r = 0; r < R; ++r) last_token[r] = -1;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0) continue;
      if (e >= E) { status = ORACLE_BAD_EXPERT_ID; continue; }
      int32_t r = (int32_t)(e / L);
      if (last_token[r] != t) { last_token[r] = t; count[r] += 1; }
    }
  }
  /* Exclusive sum over ranks: the start of each rank's block. */
  int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
  if (!cursor) return ORACLE_BAD_ARG;
  int64_t run = 0;
  for (int32_t r = 0; r < R; ++r) { cursor[r] = run; run += count[r]; }
  *total_rows = run;
  free(count);
  if (run > capacity_rows) { free(last_token); free(cursor); return ORACLE_CAPACITY; }
  /* Scatter: tokens in order; the highest k reaching rank r takes the row. */
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) rank_slot[t * K + k] = -1;
    for (int32_t k = K - 1; k >= 0; --k) {
      int64_t e = topk_idx[t * K + k];
      if (e < 0 || e >= E) continue;
      int32_t r = (int32_t)(e / L);
      int taken = 0;
      for (int32_t k2 = k + 1; k2 < K; ++k2) {
        int64_t e2 = topk_idx[t * K + k2];
        if (e2 >= 0 && e2 < E && (int32_t)(e2 / L) == r) { taken = 1; break; }
      }
      if (taken) continue;
      rank_slot[t * K + k] = (int32_t)cursor[r];
      rank_src[cursor[r]] = (int32_t)t;
      cursor[r] += 1;
    }
  }
  free(last_token);
  free(cursor);
  return status;
}

/*
 * oracle_permute -- the expand-mode row scatter ([CS] §6.4, §8.2) and the
 * zero padding of the alignment gap ([CS] §7.3).
 *
 * recv_x[dst_slot[t*K+k]] = x[t] byte for byte for every valid pair; when
 * sf is given, recv_sf rows move the same way.  With zero_pad, the rows
 * [expert_offset[e] + expert_count[e], expert_offset[e+1]) are zero bytes.
 */
int oracle_permute(int64_t N, int32_t K, const int32_t *dst_slot,
                   const uint8_t *x, int64_t row_bytes, const uint8_t *sf,
                   int64_t sf_row_bytes, int32_t E,
                   const int32_t *expert_offset, const int32_t *expert_count,
                   uint8_t *recv_x, uint8_t *recv_sf, int64_t rows,
                   int32_t zero_pad) {
  if (N < 0 || K < 1 || row_bytes < 0) return ORACLE_BAD_ARG;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int64_t s = dst_slot[t * K + k];
      if (s < 0) continue;
      if (s >= rows) return ORACLE_CAPACITY;
      memcpy(recv_x + s * row_bytes, x + t * row_bytes, (size_t)row_bytes);
      if (sf)
        memcpy(recv_sf + s * sf_row_bytes, sf + t * sf_row_bytes,
               (size_t)sf_row_bytes);
    }
  }
  if (zero_pad) {
    for (int32_t e = 0; e < E; ++e) {
      int64_t lo = (int64_t)expert_offset[e] + expert_count[e];
      int64_t hi = expert_offset[e + 1];
      for (int64_t i = lo; i < hi && i < rows; ++i) {
        memset(recv_x + i * row_bytes, 0, (size_t)row_bytes);
        if (sf) memset(recv_sf + i * sf_row_bytes, 0, (size_t)sf_row_bytes);
      }
    }
  }
  return ORACLE_OK;
}

/*
 * oracle_permute_sf_col_major -- the scale factors of the expand-mode receive
 * buffer stored column-major with a TMA-aligned leading dimension: the fetch
 * option use_tma_aligned_col_major_sf of the page "00 DeepEP Engram
 * Architecture Deep-Dive" (§1.1 Python API, §1.2 C++ runtime), cited here as
 * [EA].  [EA] names the option and defines nothing.  Reading taken: the
 * [rows, C] matrix of 4-byte scale words is stored one column after another,
 * column j at out + j*ld, and ld (the leading dimension) is a row count that
 * is a multiple of 4, so that every column starts on a 16-byte boundary as a
 * TMA global stride must.  Rows move as in oracle_permute ([CS] §6.4, §8.2):
 *   out[j*ld + dst_slot[t*K+k]] = sf[t*C + j]   for every valid pair, all j;
 * with zero_pad, rows [expert_offset[e] + expert_count[e], expert_offset[e+1])
 * are 0 in every column ([CS] §7.3).  Nothing else is written.  ld must be at
 * least `rows` (the rows the layout uses) and a multiple of 4.
 */
int oracle_permute_sf_col_major(int64_t N, int32_t K, const int32_t *dst_slot,
                                const uint32_t *sf, int64_t C, int32_t E,
                                const int32_t *expert_offset,
                                const int32_t *expert_count, uint32_t *out,
                                int64_t ld, int64_t rows, int32_t zero_pad) {
  if (N < 0 || K < 1 || C < 0 || ld < rows || ld % 4 != 0) return ORACLE_BAD_ARG;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t k = 0; k < K; ++k) {
      int64_t s = dst_slot[t * K + k];
      if (s < 0) continue;
      if (s >= rows) return ORACLE_CAPACITY;
      for (int64_t j = 0; j < C; ++j) out[j * ld + s] = sf[t * C + j];
    }
  }
  if (zero_pad) {
    for (int32_t e = 0; e < E; ++e) {
      int64_t gap_begin = (int64_t)expert_offset[e] + expert_count[e];
      int64_t gap_end = expert_offset[e + 1];
      for (int64_t i = gap_begin; i < gap_end && i < rows; ++i)
        for (int64_t j = 0; j < C; ++j) out[j * ld + i] = 0;
    }
  }
  return ORACLE_OK;
}

/* bf16 <-> fp32.  bf16 is the upper half of an IEEE binary32; widening is
   exact, narrowing rounds the dropped 16 bits to nearest, ties to even. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep it a (quiet) NaN */
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16(int64_t n, const float *in, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/*
 * oracle_expert_scale -- the stand-in "expert" of the round-trip workload:
 * row i of segment e becomes bf16(float(recv_x[i]) * scale[e]).  Pad rows
 * are zero in, zero out.  Not part of the method; it only feeds combine.
 */
void oracle_expert_scale(int64_t rows, int64_t H, const uint16_t *recv_x,
                         int32_t E, const int32_t *expert_offset,
                         const float *scale, uint16_t *eo) {
  for (int32_t e = 0; e < E; ++e) {
    for (int64_t i = expert_offset[e]; i < expert_offset[e + 1] && i < rows;
         ++i) {
      for (int64_t h = 0; h < H; ++h)
        eo[i * H + h] = f32_to_bf16_rne(bf16_to_f32(recv_x[i * H + h]) * scale[e]);
    }
  }
}

/* One token of the combine: the definition, term by term. */
static void combine_one(int64_t t, int32_t K, const int32_t *dst_slot,
                        const float *w, const uint16_t *eo, int64_t H,
                        uint16_t *out_row) {
  for (int64_t h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int32_t k = 0; k < K; ++k) {
      int64_t s = dst_slot[t * K + k];
      if (s < 0) continue;
      acc = fmaf(w[t * K + k], bf16_to_f32(eo[s * H + h]), acc);
    }
    out_row[h] = f32_to_bf16_rne(acc);
  }
}

/*
 * oracle_combine -- inverse of the dispatch: gather each token's expert
 * outputs by dst_slot and reduce them with its top-k weights.
 *   out[t, h] = bf16( sum over valid k, ascending, of w[t,k] * eo[dst_slot[t,k], h] )
 * The pages keep the slot map for the combine ([CS] §6.2) but print no
 * combine arithmetic; this is the plain definition.
 */
void oracle_combine(int64_t N, int32_t K, const int32_t *dst_slot,
                    const float *w, const uint16_t *eo, int64_t H,
                    uint16_t *out) {
  for (int64_t t = 0; t < N; ++t) combine_one(t, K, dst_slot, w, eo, H, out + t * H);
}

/* The same, for a chosen list of tokens (sampled checks at full size);
   out is [n_sel, H]. */
void oracle_combine_tokens(int64_t n_sel, const int64_t *tokens, int32_t K,
                           const int32_t *dst_slot, const float *w,
                           const uint16_t *eo, int64_t H, uint16_t *out) {
  for (int64_t i = 0; i < n_sel; ++i)
    combine_one(tokens[i], K, dst_slot, w, eo, H, out + i * H);
}
