// moe_layout_api.cu -- the extern "C" entry points of libmoe_layout.so:
// argument checks, workspace carving and kernel launches.  Semantics and
// error behaviour of each call are documented in include/moe_layout.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace moe {

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int device_sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  t_last_cuda_error = static_cast<int>(e);
  return MOE_ERR_CUDA;
}

// Identity of the calling thread's current CUDA context: cuCtxGetId of
// cuCtxGetCurrent, both reached through the runtime's driver entry points (no
// link-time dependency on the driver library).  0 when there is no current
// context yet or the driver lacks the calls; callers then skip their caches.
uint64_t current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id) + 1;   // never 0 for a real context
}

namespace {
struct SmemLimit {
  uint64_t ctx;
  const void* func;
  size_t bytes;
};
std::mutex g_smem_mu;
std::vector<SmemLimit> g_smem_limits;
}  // namespace

cudaError_t ensure_smem_limit(const void* func, size_t smem) {
  // Launches within the default 48 KB need no attribute.
  if (smem <= 48 * 1024) return cudaSuccess;
  const uint64_t ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_smem_mu);
    for (const SmemLimit& l : g_smem_limits)
      if (l.ctx == ctx && l.func == func && l.bytes >= smem) return cudaSuccess;
  }
  const cudaError_t st = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (st != cudaSuccess || ctx == 0) return st;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (SmemLimit& l : g_smem_limits)
    if (l.ctx == ctx && l.func == func) {
      if (smem > l.bytes) l.bytes = smem;
      return cudaSuccess;
    }
  g_smem_limits.push_back(SmemLimit{ctx, func, smem});
  return cudaSuccess;
}

namespace {
struct Occupancy {
  int dev;
  const void* func;
  int threads;
  size_t smem;
  int ctas;
};
std::mutex g_occ_mu;
std::vector<Occupancy> g_occ;
}  // namespace

int cached_occupancy(const void* func, int threads, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (const Occupancy& o : g_occ)
      if (o.dev == dev && o.func == func && o.threads == threads && o.smem == smem) return o.ctas;
  }
  int n = 0;
  if (ensure_smem_limit(func, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem) != cudaSuccess)
    return 0;   // not cached: the next call asks again
  std::lock_guard<std::mutex> lock(g_occ_mu);
  if (g_occ.size() < 256) g_occ.push_back(Occupancy{dev, func, threads, smem, n});
  return n;
}

bool cooperative_launch_supported() {
  static std::mutex mu;
  static std::vector<int> cache;   // per device: 0 unknown, 1 no, 2 yes
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) return false;
    cache[dev] = coop ? 2 : 1;
  }
  return cache[dev] == 2;
}

static std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
static std::atomic<unsigned> g_barrier_extra{0};
static std::atomic<unsigned> g_extra_tx{0};

WaitConfig wait_config() {
  return WaitConfig{g_wait_limit_ns.load(std::memory_order_relaxed), g_barrier_extra.load(std::memory_order_relaxed),
                    g_extra_tx.load(std::memory_order_relaxed)};
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_desc(const moe_layout_desc* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->num_tokens < 0 || d->topk < 1 || d->num_experts < 1 || d->num_ranks < 1 || d->alignment < 1)
    return MOE_ERR_INVALID_ARG;
  if (d->num_experts % d->num_ranks != 0) return MOE_ERR_INVALID_ARG;
  if (d->topk > MOE_MAX_TOPK || d->num_experts > MOE_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
  // Every slot and row index must fit int32.  N is bounded first, so that
  // N * K is only formed when it cannot overflow.
  if (d->num_tokens > (int64_t{1} << 31) / d->topk) return MOE_ERR_UNSUPPORTED;
  const int64_t worst = d->num_tokens * d->topk + static_cast<int64_t>(d->num_experts) * (d->alignment - 1);
  if (worst >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_workspace(const moe_layout_desc* d, const void* ws, size_t ws_bytes, WorkspaceLayout* out) {
  const WorkspaceLayout w = make_workspace_layout(*d, make_tile_plan(d->num_tokens, d->topk));
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < w.bytes) return MOE_ERR_INVALID_ARG;
  *out = w;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_layout_workspace_bytes(const moe_layout_desc* desc, size_t* bytes) {
  if (int st = check_desc(desc)) return st;
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_workspace_layout(*desc, make_tile_plan(desc->num_tokens, desc->topk)).bytes;
  return MOE_OK;
}

int moe_layout_count(const moe_layout_desc* desc, const int64_t* topk_idx, int32_t* expert_count,
                     int32_t* rank_count, void* workspace, size_t workspace_bytes, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  if ((desc->num_tokens > 0 && topk_idx == nullptr) || expert_count == nullptr || rank_count == nullptr)
    return MOE_ERR_INVALID_ARG;
  const TilePlan p = make_tile_plan(desc->num_tokens, desc->topk);
  return cuda_status(launch_count(*desc, p, IdsRef{topk_idx, false}, expert_count, rank_count, at<int>(workspace, w.err_off),
                                  at<int32_t>(workspace, w.hist_off), at<int32_t>(workspace, w.rhist_off),
                                  static_cast<cudaStream_t>(stream)));
}

int moe_layout_scan(const moe_layout_desc* desc, const int64_t* topk_idx, const int32_t* expert_count,
                    const int32_t* rank_count, void* workspace, size_t workspace_bytes,
                    int32_t* expert_offset, int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx,
                    int64_t capacity_rows, int32_t* total_rows, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  const bool has_pairs = desc->num_tokens > 0;
  if ((has_pairs && (topk_idx == nullptr || dst_slot == nullptr)) || expert_count == nullptr ||
      rank_count == nullptr || expert_offset == nullptr || rank_psum == nullptr || total_rows == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (capacity_rows < 0 || (capacity_rows > 0 && src_idx == nullptr)) return MOE_ERR_INVALID_ARG;
  const TilePlan p = make_tile_plan(desc->num_tokens, desc->topk);
  return cuda_status(launch_rank(*desc, p, IdsRef{topk_idx, false}, at<int32_t>(workspace, w.hist_off), expert_count,
                                 rank_count, expert_offset, rank_psum, dst_slot, src_idx, capacity_rows,
                                 total_rows, at<int>(workspace, w.err_off), static_cast<cudaStream_t>(stream)));
}

static int build_impl(const moe_layout_desc* desc, IdsRef ids, int32_t* expert_count, int32_t* rank_count,
                      void* workspace, size_t workspace_bytes, int32_t* expert_offset, int32_t* rank_psum,
                      int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows, int32_t* total_rows,
                      void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  const bool has_pairs = desc->num_tokens > 0;
  if ((has_pairs && (ids.ptr == nullptr || dst_slot == nullptr)) || expert_count == nullptr ||
      rank_count == nullptr || expert_offset == nullptr || rank_psum == nullptr || total_rows == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (capacity_rows < 0 || (capacity_rows > 0 && src_idx == nullptr)) return MOE_ERR_INVALID_ARG;
  const TilePlan p = make_tile_plan(desc->num_tokens, desc->topk);
  return cuda_status(launch_build(*desc, p, ids, expert_count, rank_count, at<int32_t>(workspace, w.hist_off),
                                  at<int32_t>(workspace, w.rhist_off), at<unsigned>(workspace, w.bar_off),
                                  expert_offset, rank_psum, dst_slot, src_idx, capacity_rows, total_rows,
                                  at<int>(workspace, w.err_off), static_cast<cudaStream_t>(stream)));
}

int moe_layout_build(const moe_layout_desc* desc, const int64_t* topk_idx, int32_t* expert_count,
                     int32_t* rank_count, void* workspace, size_t workspace_bytes, int32_t* expert_offset,
                     int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                     int32_t* total_rows, void* stream) {
  return build_impl(desc, IdsRef{topk_idx, false}, expert_count, rank_count, workspace, workspace_bytes,
                    expert_offset, rank_psum, dst_slot, src_idx, capacity_rows, total_rows, stream);
}

int moe_layout_build_i32(const moe_layout_desc* desc, const int32_t* topk_idx, int32_t* expert_count,
                         int32_t* rank_count, void* workspace, size_t workspace_bytes, int32_t* expert_offset,
                         int32_t* rank_psum, int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                         int32_t* total_rows, void* stream) {
  return build_impl(desc, IdsRef{topk_idx, true}, expert_count, rank_count, workspace, workspace_bytes,
                    expert_offset, rank_psum, dst_slot, src_idx, capacity_rows, total_rows, stream);
}

int moe_dispatch_permute(const moe_layout_desc* desc, const void* x, int64_t row_bytes, const void* sf,
                         int64_t sf_row_bytes, const int32_t* dst_slot, const int32_t* expert_offset,
                         const int32_t* expert_count, void* recv_x, void* recv_sf, int64_t capacity_rows,
                         int zero_pad, void* workspace, size_t workspace_bytes, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  const bool has_pairs = desc->num_tokens > 0;
  if (row_bytes <= 0 || row_bytes % 16 != 0 || capacity_rows < 0) return MOE_ERR_INVALID_ARG;
  if ((has_pairs && (x == nullptr || dst_slot == nullptr)) || expert_offset == nullptr ||
      expert_count == nullptr || (capacity_rows > 0 && recv_x == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16)) return MOE_ERR_INVALID_ARG;
  if (sf != nullptr) {
    if (sf_row_bytes <= 0 || sf_row_bytes % 4 != 0 || !aligned(sf, 4) || !aligned(recv_sf, 4) ||
        (capacity_rows > 0 && recv_sf == nullptr))
      return MOE_ERR_INVALID_ARG;
  }
  if (row_bytes > MOE_MAX_ROW_BYTES || (sf != nullptr && sf_row_bytes > MOE_MAX_ROW_BYTES)) return MOE_ERR_UNSUPPORTED;
  PermuteArgs a{};
  a.x = static_cast<const uint8_t*>(x);
  a.sf = static_cast<const uint8_t*>(sf);
  a.row_bytes = row_bytes;
  a.sf_row_bytes = sf != nullptr ? sf_row_bytes : 0;
  a.dst_slot = dst_slot;
  a.total_rows = expert_offset + desc->num_experts;
  a.expert_offset = expert_offset;
  a.expert_count = expert_count;
  a.recv_x = static_cast<uint8_t*>(recv_x);
  a.recv_sf = sf != nullptr ? static_cast<uint8_t*>(recv_sf) : nullptr;
  a.capacity = capacity_rows;
  a.num_tokens = desc->num_tokens;
  a.topk = desc->topk;
  a.num_experts = desc->num_experts;
  a.zero_pad = zero_pad != 0;
  a.err = at<int>(workspace, w.err_off);
  a.work = at<unsigned>(workspace, w.work_off);
  return cuda_status(launch_permute(a, static_cast<cudaStream_t>(stream)));
}

int moe_layout_rank_rows(const moe_layout_desc* desc, const int64_t* topk_idx, const int32_t* rank_count,
                         void* workspace, size_t workspace_bytes, int32_t* rank_slot, int32_t* rank_src,
                         int64_t capacity_rows, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  const bool has_pairs = desc->num_tokens > 0;
  if ((has_pairs && (topk_idx == nullptr || rank_slot == nullptr)) || rank_count == nullptr) return MOE_ERR_INVALID_ARG;
  if (capacity_rows < 0 || (capacity_rows > 0 && rank_src == nullptr)) return MOE_ERR_INVALID_ARG;
  const TilePlan p = make_tile_plan(desc->num_tokens, desc->topk);
  return cuda_status(launch_rank_rows(*desc, p, IdsRef{topk_idx, false}, at<int32_t>(workspace, w.rhist_off), rank_count, rank_slot,
                                      rank_src, capacity_rows, at<int>(workspace, w.err_off),
                                      static_cast<cudaStream_t>(stream)));
}

int moe_dispatch_permute_ranks(const moe_layout_desc* desc, const void* x, int64_t row_bytes, const void* sf,
                               int64_t sf_row_bytes, const int32_t* rank_slot, const int32_t* rank_psum,
                               void* recv, void* recv_sf, int64_t capacity_rows, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  const bool has_pairs = desc->num_tokens > 0;
  if (row_bytes <= 0 || row_bytes % 16 != 0 || capacity_rows < 0) return MOE_ERR_INVALID_ARG;
  if ((has_pairs && (x == nullptr || rank_slot == nullptr)) || rank_psum == nullptr ||
      (capacity_rows > 0 && recv == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv, 16)) return MOE_ERR_INVALID_ARG;
  if (sf != nullptr) {
    if (sf_row_bytes <= 0 || sf_row_bytes % 4 != 0 || !aligned(sf, 4) || !aligned(recv_sf, 4) ||
        (capacity_rows > 0 && recv_sf == nullptr))
      return MOE_ERR_INVALID_ARG;
  }
  if (row_bytes > MOE_MAX_ROW_BYTES || (sf != nullptr && sf_row_bytes > MOE_MAX_ROW_BYTES)) return MOE_ERR_UNSUPPORTED;
  PermuteArgs a{};
  a.x = static_cast<const uint8_t*>(x);
  a.sf = static_cast<const uint8_t*>(sf);
  a.row_bytes = row_bytes;
  a.sf_row_bytes = sf != nullptr ? sf_row_bytes : 0;
  a.dst_slot = rank_slot;
  a.total_rows = rank_psum + (desc->num_ranks - 1);
  a.expert_offset = nullptr;
  a.expert_count = nullptr;
  a.recv_x = static_cast<uint8_t*>(recv);
  a.recv_sf = sf != nullptr ? static_cast<uint8_t*>(recv_sf) : nullptr;
  a.capacity = capacity_rows;
  a.num_tokens = desc->num_tokens;
  a.topk = desc->topk;
  a.num_experts = desc->num_experts;
  a.zero_pad = 0;
  a.err = at<int>(workspace, w.err_off);
  a.work = at<unsigned>(workspace, w.work_off);
  a.non_expand = true;
  return cuda_status(launch_permute(a, static_cast<cudaStream_t>(stream)));
}

int moe_dispatch_sf_col_major(const moe_layout_desc* desc, const void* sf, int64_t sf_cols, const int32_t* src,
                              const int32_t* total_rows, void* recv_sf_cm, int64_t ld, int64_t capacity_rows,
                              int zero_pad, void* workspace, size_t workspace_bytes, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  if (sf_cols <= 0 || capacity_rows < 0 || ld < capacity_rows || ld % 4 != 0 || total_rows == nullptr)
    return MOE_ERR_INVALID_ARG;
  if ((desc->num_tokens > 0 && sf == nullptr) || (capacity_rows > 0 && (src == nullptr || recv_sf_cm == nullptr)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(sf, 4) || !aligned(recv_sf_cm, 16)) return MOE_ERR_INVALID_ARG;
  if (sf_cols > MOE_MAX_ROW_BYTES / 4 || ld > (int64_t{1} << 32)) return MOE_ERR_UNSUPPORTED;
  SfColMajorArgs a{};
  a.sf = static_cast<const uint32_t*>(sf);
  a.cols = sf_cols;
  a.src = src;
  a.total_rows = total_rows;
  a.out = static_cast<uint32_t*>(recv_sf_cm);
  a.ld = ld;
  a.capacity = capacity_rows;
  a.num_tokens = desc->num_tokens;
  a.zero_pad = zero_pad != 0;
  a.err = at<int>(workspace, w.err_off);
  return cuda_status(launch_sf_col_major(a, static_cast<cudaStream_t>(stream)));
}

int moe_combine_unpermute(const moe_layout_desc* desc, const void* expert_out, int64_t expert_out_rows,
                          int64_t hidden, const int32_t* dst_slot, const float* weights, void* out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (int st = check_desc(desc)) return st;
  WorkspaceLayout w;
  if (int st = check_workspace(desc, workspace, workspace_bytes, &w)) return st;
  if (hidden <= 0 || hidden % 8 != 0 || expert_out_rows < 0) return MOE_ERR_INVALID_ARG;
  if (hidden > MOE_MAX_ROW_BYTES / 2) return MOE_ERR_UNSUPPORTED;
  if (desc->num_tokens == 0) return MOE_OK;
  if (dst_slot == nullptr || weights == nullptr || out == nullptr ||
      (expert_out_rows > 0 && expert_out == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(weights, 4)) return MOE_ERR_INVALID_ARG;
  CombineArgs a{};
  a.expert_out = static_cast<const uint16_t*>(expert_out);
  a.expert_out_rows = expert_out_rows;
  a.hidden = hidden;
  a.dst_slot = dst_slot;
  a.weights = weights;
  a.out = static_cast<uint16_t*>(out);
  a.num_tokens = desc->num_tokens;
  a.topk = desc->topk;
  a.err = at<int>(workspace, w.err_off);
  a.work = at<unsigned>(workspace, w.work_off) + 2;
  return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

int moe_layout_accumulate_stats(const moe_layout_desc* desc, const int32_t* expert_count, int64_t* cumulative,
                                void* stream) {
  if (int st = check_desc(desc)) return st;
  if (expert_count == nullptr || cumulative == nullptr || !aligned(cumulative, 8)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_accumulate_stats(expert_count, desc->num_experts, cumulative,
                                             static_cast<cudaStream_t>(stream)));
}

int moe_layout_get_error(void* workspace, int32_t* device_error, void* stream) {
  if (workspace == nullptr || device_error == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  *device_error = host;
  return MOE_OK;
}

const char* moe_strerror(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id >= num_experts";
    case MOE_ERR_CAPACITY: return "receive buffer capacity exceeded";
    case MOE_ERR_TIMEOUT: return "bounded wait in a kernel timed out";
    case MOE_ERR_UNSUPPORTED: return "sizes beyond this build's limits";
    default: return "unknown status";
  }
}

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_debug_set_waits(uint64_t limit_ns, uint32_t barrier_extra, uint32_t extra_tx) {
  if (limit_ns > kWaitLimitNs || extra_tx % 16 != 0) return MOE_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns, std::memory_order_relaxed);
  g_barrier_extra.store(barrier_extra, std::memory_order_relaxed);
  g_extra_tx.store(extra_tx, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_last_cuda_error(const char** message) {
  if (message != nullptr) *message = cudaGetErrorString(static_cast<cudaError_t>(t_last_cuda_error));
  return t_last_cuda_error;
}

}  // extern "C"
