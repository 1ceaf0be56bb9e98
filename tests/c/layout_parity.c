/*
 * GPU parity through the C ABI alone: no Python, no PyTorch on the data path.
 *
 * For each case: seeded routing ids (distinct experts per token, some slots
 * masked), token rows and weights are drawn here; the library runs
 * moe_layout_build, moe_dispatch_permute and moe_combine_unpermute (with the
 * receive rows standing in for the expert outputs) on device memory from the
 * CUDA runtime, on the legacy default stream; the oracle (oracle/oracle.c,
 * linked into this test) computes the same from the same inputs on the CPU.
 * Every output is compared bit for bit.  Exit status 0 means all cases match.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe_layout.h"

/* oracle/oracle.c */
int oracle_layout(int64_t N, int32_t K, int32_t E, int32_t R, int32_t A, const int64_t *topk_idx,
                  int32_t *expert_count, int32_t *rank_count, int32_t *expert_offset, int32_t *rank_psum,
                  int32_t *dst_slot, int32_t *src_idx, int64_t capacity_rows, int64_t *total_rows);
int oracle_permute(int64_t N, int32_t K, const int32_t *dst_slot, const uint8_t *x, int64_t row_bytes,
                   const uint8_t *sf, int64_t sf_row_bytes, int32_t E, const int32_t *expert_offset,
                   const int32_t *expert_count, uint8_t *recv_x, uint8_t *recv_sf, int64_t rows, int32_t zero_pad);
void oracle_combine(int64_t N, int32_t K, const int32_t *dst_slot, const float *w, const uint16_t *eo, int64_t H,
                    uint16_t *out);

/* splitmix64: a counter-based generator for the inputs */
static uint64_t mix(uint64_t *s) {
  uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

#define CHECK_CUDA(call)                                                                  \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) {                                                              \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
      return 10;                                                                          \
    }                                                                                     \
  } while (0)
#define CHECK_MOE(call)                                                                   \
  do {                                                                                    \
    int s_ = (call);                                                                      \
    if (s_ != MOE_OK) {                                                                   \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #call, moe_strerror(s_));     \
      return 11;                                                                          \
    }                                                                                     \
  } while (0)

static int same(const char *what, const void *a, const void *b, size_t bytes) {
  if (bytes == 0 || memcmp(a, b, bytes) == 0) return 1;
  fprintf(stderr, "mismatch: %s\n", what);
  return 0;
}

static int run_case(int64_t N, int32_t K, int32_t E, int32_t R, int32_t A, int64_t H, uint64_t seed,
                    unsigned mask_per_mille) {
  const int64_t rb = H * 2; /* bf16 rows */
  const int64_t cap = N * K + (int64_t)E * (A - 1);
  const int64_t pairs = N * K;
  moe_layout_desc d;
  memset(&d, 0, sizeof d);
  d.num_tokens = N; d.topk = K; d.num_experts = E; d.num_ranks = R; d.alignment = A;

  /* inputs */
  int64_t *idx = malloc(sizeof(int64_t) * (size_t)(pairs ? pairs : 1));
  uint16_t *x = malloc((size_t)(N ? N : 1) * (size_t)rb);
  float *w = malloc(sizeof(float) * (size_t)(pairs ? pairs : 1));
  int32_t *perm = malloc(sizeof(int32_t) * (size_t)E);
  uint64_t s = seed;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t e = 0; e < E; ++e) perm[e] = e;
    for (int32_t k = 0; k < K; ++k) { /* partial Fisher-Yates: distinct experts */
      const int32_t j = k + (int32_t)(mix(&s) % (uint64_t)(E - k));
      const int32_t tmp = perm[k]; perm[k] = perm[j]; perm[j] = tmp;
      idx[t * K + k] = (mix(&s) % 1000u) < mask_per_mille ? -1 : perm[k];
      w[t * K + k] = (float)(mix(&s) >> 40) / (float)(1u << 24);
    }
    for (int64_t h = 0; h < H; ++h) { /* finite bf16: exponent away from all-ones */
      const uint64_t r = mix(&s);
      x[t * H + h] = (uint16_t)(((r & 0x8000u) | (0x3000u + (r >> 16) % 0x1000u)) & 0xffffu);
    }
  }

  /* oracle */
  int32_t *o_ec = calloc((size_t)E, 4), *o_rc = calloc((size_t)R, 4), *o_off = calloc((size_t)E + 1, 4);
  int32_t *o_ps = calloc((size_t)R, 4), *o_dst = calloc((size_t)(pairs ? pairs : 1), 4);
  int32_t *o_src = calloc((size_t)(cap ? cap : 1), 4);
  int64_t o_rows = 0;
  if (oracle_layout(N, K, E, R, A, idx, o_ec, o_rc, o_off, o_ps, o_dst, o_src, cap, &o_rows) != 0) return 20;
  uint8_t *o_recv = calloc((size_t)(o_rows ? o_rows : 1), (size_t)rb);
  if (oracle_permute(N, K, o_dst, (const uint8_t *)x, rb, NULL, 0, E, o_off, o_ec, o_recv, NULL, o_rows, 1) != 0)
    return 21;
  uint16_t *o_out = calloc((size_t)(N ? N : 1), (size_t)rb);
  oracle_combine(N, K, o_dst, w, (const uint16_t *)o_recv, H, o_out);

  /* library */
  size_t ws_bytes = 0;
  CHECK_MOE(moe_layout_workspace_bytes(&d, &ws_bytes));
  void *ws, *d_x, *d_recv, *d_out;
  int64_t *d_idx;
  float *d_w;
  int32_t *d_ec, *d_rc, *d_off, *d_ps, *d_dst, *d_src, *d_rows;
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemset(ws, 0, ws_bytes)); /* zero-filled once before first use */
  CHECK_CUDA(cudaMalloc((void **)&d_idx, sizeof(int64_t) * (size_t)(pairs ? pairs : 1)));
  CHECK_CUDA(cudaMalloc(&d_x, (size_t)(N ? N : 1) * (size_t)rb));
  CHECK_CUDA(cudaMalloc((void **)&d_w, sizeof(float) * (size_t)(pairs ? pairs : 1)));
  CHECK_CUDA(cudaMalloc((void **)&d_ec, 4 * (size_t)E));
  CHECK_CUDA(cudaMalloc((void **)&d_rc, 4 * (size_t)R));
  CHECK_CUDA(cudaMalloc((void **)&d_off, 4 * ((size_t)E + 1)));
  CHECK_CUDA(cudaMalloc((void **)&d_ps, 4 * (size_t)R));
  CHECK_CUDA(cudaMalloc((void **)&d_dst, 4 * (size_t)(pairs ? pairs : 1)));
  CHECK_CUDA(cudaMalloc((void **)&d_src, 4 * (size_t)(cap ? cap : 1)));
  CHECK_CUDA(cudaMalloc((void **)&d_rows, 4));
  CHECK_CUDA(cudaMalloc(&d_recv, (size_t)(cap ? cap : 1) * (size_t)rb));
  CHECK_CUDA(cudaMalloc(&d_out, (size_t)(N ? N : 1) * (size_t)rb));
  CHECK_CUDA(cudaMemcpy(d_idx, idx, sizeof(int64_t) * (size_t)pairs, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(d_x, x, (size_t)N * (size_t)rb, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(d_w, w, sizeof(float) * (size_t)pairs, cudaMemcpyHostToDevice));
  CHECK_MOE(moe_layout_build(&d, d_idx, d_ec, d_rc, ws, ws_bytes, d_off, d_ps, d_dst, d_src, cap, d_rows, NULL));
  CHECK_MOE(moe_dispatch_permute(&d, d_x, rb, NULL, 0, d_dst, d_off, d_ec, d_recv, NULL, cap, 1, ws, ws_bytes, NULL));
  CHECK_MOE(moe_combine_unpermute(&d, d_recv, cap, H, d_dst, d_w, d_out, ws, ws_bytes, NULL));
  int32_t dev_err = -1;
  CHECK_MOE(moe_layout_get_error(ws, &dev_err, NULL)); /* synchronises the stream */
  if (dev_err != MOE_OK) {
    fprintf(stderr, "device error %d: %s\n", dev_err, moe_strerror(dev_err));
    return 12;
  }

  int32_t g_rows = -1;
  int32_t *g_ec = malloc(4 * (size_t)E), *g_rc = malloc(4 * (size_t)R), *g_off = malloc(4 * ((size_t)E + 1));
  int32_t *g_ps = malloc(4 * (size_t)R), *g_dst = malloc(4 * (size_t)(pairs ? pairs : 1));
  int32_t *g_src = malloc(4 * (size_t)(o_rows ? o_rows : 1));
  uint8_t *g_recv = malloc((size_t)(o_rows ? o_rows : 1) * (size_t)rb);
  uint16_t *g_out = malloc((size_t)(N ? N : 1) * (size_t)rb);
  CHECK_CUDA(cudaMemcpy(&g_rows, d_rows, 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_ec, d_ec, 4 * (size_t)E, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_rc, d_rc, 4 * (size_t)R, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_off, d_off, 4 * ((size_t)E + 1), cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_ps, d_ps, 4 * (size_t)R, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_dst, d_dst, 4 * (size_t)pairs, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_src, d_src, 4 * (size_t)o_rows, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_recv, d_recv, (size_t)o_rows * (size_t)rb, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(g_out, d_out, (size_t)N * (size_t)rb, cudaMemcpyDeviceToHost));

  int ok = g_rows == o_rows;
  if (!ok) fprintf(stderr, "mismatch: total_rows %d vs %lld\n", g_rows, (long long)o_rows);
  ok &= same("expert_count", g_ec, o_ec, 4 * (size_t)E);
  ok &= same("rank_count", g_rc, o_rc, 4 * (size_t)R);
  ok &= same("expert_offset", g_off, o_off, 4 * ((size_t)E + 1));
  ok &= same("rank_psum", g_ps, o_ps, 4 * (size_t)R);
  ok &= same("dst_slot", g_dst, o_dst, 4 * (size_t)pairs);
  ok &= same("src_idx", g_src, o_src, 4 * (size_t)o_rows);
  ok &= same("recv_x", g_recv, o_recv, (size_t)o_rows * (size_t)rb);
  ok &= same("combine out", g_out, o_out, (size_t)N * (size_t)rb);
  printf("N=%lld K=%d E=%d R=%d A=%d H=%lld rows=%lld %s\n", (long long)N, K, E, R, A, (long long)H,
         (long long)o_rows, ok ? "match" : "MISMATCH");

  cudaFree(ws); cudaFree(d_x); cudaFree(d_recv); cudaFree(d_out); cudaFree(d_idx); cudaFree(d_w);
  cudaFree(d_ec); cudaFree(d_rc); cudaFree(d_off); cudaFree(d_ps); cudaFree(d_dst); cudaFree(d_src);
  cudaFree(d_rows);
  free(idx); free(x); free(w); free(perm); free(o_ec); free(o_rc); free(o_off); free(o_ps); free(o_dst);
  free(o_src); free(o_recv); free(o_out); free(g_ec); free(g_rc); free(g_off); free(g_ps); free(g_dst);
  free(g_src); free(g_recv); free(g_out);
  return ok ? 0 : 1;
}

int main(void) {
  int st = 0;
  if ((st = run_case(4096, 8, 256, 8, 128, 7168, 1, 0)) != 0) return st;   /* decode: 4096 x top-8, 7168 bf16 */
  if ((st = run_case(1000, 3, 40, 5, 16, 64, 2, 100)) != 0) return st;     /* ragged tiles, 10 % masked */
  if ((st = run_case(40007, 3, 40, 5, 16, 16, 3, 50)) != 0) return st;     /* the cooperative layout kernel */
  if ((st = run_case(0, 8, 16, 4, 8, 64, 4, 0)) != 0) return st;           /* empty batch */
  printf("all cases match\n");
  return 0;
}
