// host_pipeline.cu -- dispatch from host memory and combine to host memory,
// with the host<->device copies overlapped with the kernels.
//
// moe_dispatch_from_host: ids (and weights) first, then the layout, while
// the token rows stream to the device in chunks on a copy stream; each
// chunk's permute starts as soon as its rows have landed.
// moe_combine_to_host: the combine runs chunk by chunk and each chunk's
// result is copied back while the next chunk is combined.
//
// Both are orchestration only: every step of the computation is one of the
// library's other entry points (moe_layout_build, moe_dispatch_permute,
// moe_combine_unpermute) applied to a token range through offset pointers.
#include <cuda_runtime.h>

#include "common.cuh"

namespace {

// One event serves every hand-off in a call: a wait captures the event's
// state when it is enqueued, so the event can be recorded again right after.
struct CallEvent {
  cudaEvent_t ev = nullptr;
  cudaError_t st = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  ~CallEvent() {
    if (ev != nullptr) cudaEventDestroy(ev);   // released once pending work completes
  }
};

// `waiter` waits for everything enqueued on `signaler` so far.
cudaError_t order_after(cudaEvent_t ev, cudaStream_t signaler, cudaStream_t waiter) {
  cudaError_t st = cudaEventRecord(ev, signaler);
  if (st == cudaSuccess) st = cudaStreamWaitEvent(waiter, ev, 0);
  return st;
}

int64_t chunk_size(int64_t n, int64_t chunk_tokens) { return chunk_tokens > 0 ? chunk_tokens : (n > 0 ? n : 1); }

}  // namespace

extern "C" int moe_dispatch_from_host(const moe_layout_desc* desc, const int64_t* topk_idx_host,
                                      const void* x_host, int64_t row_bytes, const void* sf_host,
                                      int64_t sf_row_bytes, const float* weights_host, int64_t* topk_idx,
                                      void* x, void* sf, float* weights, int32_t* expert_count,
                                      int32_t* rank_count, int32_t* expert_offset, int32_t* rank_psum,
                                      int32_t* dst_slot, int32_t* src_idx, int32_t* total_rows, void* recv_x,
                                      void* recv_sf, int64_t capacity_rows, void* workspace,
                                      size_t workspace_bytes, int64_t chunk_tokens, void* stream,
                                      void* copy_stream) {
  size_t need = 0;
  if (int st = moe_layout_workspace_bytes(desc, &need)) return st;
  const int64_t N = desc->num_tokens;
  const int K = desc->topk;
  if (N > 0 && (topk_idx_host == nullptr || x_host == nullptr || topk_idx == nullptr || x == nullptr))
    return MOE_ERR_INVALID_ARG;
  if ((weights_host == nullptr) != (weights == nullptr) || (sf_host == nullptr) != (sf == nullptr) ||
      row_bytes <= 0 || chunk_tokens < 0)
    return MOE_ERR_INVALID_ARG;
  if (row_bytes > MOE_MAX_ROW_BYTES || (sf_host != nullptr && sf_row_bytes > MOE_MAX_ROW_BYTES))
    return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  CallEvent e;
  if (e.st != cudaSuccess) return moe::cuda_status(e.st);
  // The staging buffers may still be read by earlier work on `stream`.
  if (cudaError_t ce = order_after(e.ev, s, cs)) return moe::cuda_status(ce);
  if (N > 0) {
    if (cudaError_t ce = cudaMemcpyAsync(topk_idx, topk_idx_host, sizeof(int64_t) * N * K, cudaMemcpyHostToDevice, s))
      return moe::cuda_status(ce);
  }
  if (weights != nullptr && N > 0) {
    if (cudaError_t ce = cudaMemcpyAsync(weights, weights_host, sizeof(float) * N * K, cudaMemcpyHostToDevice, cs))
      return moe::cuda_status(ce);
  }
  if (int st = moe_layout_build(desc, topk_idx, expert_count, rank_count, workspace, workspace_bytes, expert_offset,
                                rank_psum, dst_slot, src_idx, capacity_rows, total_rows, stream))
    return st;
  const int64_t C = chunk_size(N, chunk_tokens);
  for (int64_t t0 = 0; t0 < N || t0 == 0; t0 += C) {
    const int64_t n = N > t0 ? (N - t0 < C ? N - t0 : C) : 0;
    if (n > 0) {
      const uint8_t* xh = static_cast<const uint8_t*>(x_host) + t0 * row_bytes;
      uint8_t* xd = static_cast<uint8_t*>(x) + t0 * row_bytes;
      if (cudaError_t ce = cudaMemcpyAsync(xd, xh, static_cast<size_t>(n * row_bytes), cudaMemcpyHostToDevice, cs))
        return moe::cuda_status(ce);
      if (sf != nullptr) {
        if (cudaError_t ce = cudaMemcpyAsync(static_cast<uint8_t*>(sf) + t0 * sf_row_bytes,
                                             static_cast<const uint8_t*>(sf_host) + t0 * sf_row_bytes,
                                             static_cast<size_t>(n * sf_row_bytes), cudaMemcpyHostToDevice, cs))
          return moe::cuda_status(ce);
      }
    }
    if (cudaError_t ce = order_after(e.ev, cs, s)) return moe::cuda_status(ce);
    moe_layout_desc part = *desc;
    part.num_tokens = n;
    // The first chunk's launch also zero-fills every gap row of the buffer.
    const int zero_pad = t0 == 0 ? 1 : 0;
    if (int st = moe_dispatch_permute(&part, static_cast<uint8_t*>(x) + t0 * row_bytes, row_bytes,
                                      sf != nullptr ? static_cast<uint8_t*>(sf) + t0 * sf_row_bytes : nullptr,
                                      sf_row_bytes, dst_slot + t0 * K, expert_offset, expert_count, recv_x,
                                      recv_sf, capacity_rows, zero_pad, workspace, workspace_bytes, stream))
      return st;
    if (N == 0) break;
  }
  return MOE_OK;
}

extern "C" int moe_combine_to_host(const moe_layout_desc* desc, const void* expert_out, int64_t expert_out_rows,
                                   int64_t hidden, const int32_t* dst_slot, const float* weights, void* out,
                                   void* out_host, void* workspace, size_t workspace_bytes, int64_t chunk_tokens,
                                   void* stream, void* copy_stream) {
  size_t need = 0;
  if (int st = moe_layout_workspace_bytes(desc, &need)) return st;
  const int64_t N = desc->num_tokens;
  const int K = desc->topk;
  if ((N > 0 && (out == nullptr || out_host == nullptr)) || hidden <= 0 || chunk_tokens < 0)
    return MOE_ERR_INVALID_ARG;
  if (hidden > MOE_MAX_ROW_BYTES / 2) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
  CallEvent e;
  if (e.st != cudaSuccess) return moe::cuda_status(e.st);
  // The host buffer may still be the target of earlier copies on copy_stream.
  if (cudaError_t ce = order_after(e.ev, cs, s)) return moe::cuda_status(ce);
  const int64_t C = chunk_size(N, chunk_tokens);
  const size_t row = static_cast<size_t>(hidden) * 2;   // bf16
  for (int64_t t0 = 0; t0 < N; t0 += C) {
    const int64_t n = N - t0 < C ? N - t0 : C;
    moe_layout_desc part = *desc;
    part.num_tokens = n;
    if (int st = moe_combine_unpermute(&part, expert_out, expert_out_rows, hidden, dst_slot + t0 * K,
                                       weights + t0 * K, static_cast<uint8_t*>(out) + t0 * row, workspace,
                                       workspace_bytes, stream))
      return st;
    if (cudaError_t ce = order_after(e.ev, s, cs)) return moe::cuda_status(ce);
    if (cudaError_t ce = cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + t0 * row,
                                         static_cast<uint8_t*>(out) + t0 * row, static_cast<size_t>(n) * row,
                                         cudaMemcpyDeviceToHost, cs))
      return moe::cuda_status(ce);
  }
  // Work enqueued on `stream` afterwards (or a synchronize of it) sees the copies done.
  if (cudaError_t ce = order_after(e.ev, cs, s)) return moe::cuda_status(ce);
  return MOE_OK;
}
