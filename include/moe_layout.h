/*
 * moe_layout.h -- C ABI of the GB300 MoE dispatch-layout library
 * (libmoe_layout.so): token dispatch as a counting sort / bucketization,
 * and its inverse combine, on one GPU.
 *
 * The method is the one described on the page
 *   "07 DeepEP Counting Sort / Bucketization 深度校验：博客第一性原理 vs 源码实现"
 * cited as [CS] with its section numbers: count tokens per expert and per
 * logical rank (§4.2), prefix-sum the aligned counts (§5.2-§5.5, §7.2),
 * scatter every (token, expert) copy of a row into an expert-major buffer
 * (§6.4, §8.2) with zero rows in the alignment gaps (§7.3).  Combine is the
 * inverse gather with a top-k weighted sum.
 *
 * Conventions shared by every entry point
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory; scratch lives in a caller-provided workspace whose
 *    size moe_layout_workspace_bytes() returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and returns before the GPU work finishes, except
 *    moe_layout_get_error(), which synchronises the stream.
 *  - Return value: MOE_OK, or an error found on the host before anything was
 *    launched (MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED), or MOE_ERR_CUDA if a
 *    launch failed.  Errors found by the kernels (bad expert id, capacity,
 *    timeout, an inverse-map entry out of range) are recorded in the
 *    workspace's sticky error word and read with moe_layout_get_error().
 *  - Notation: N tokens, K top-k slots, E experts, R logical ranks,
 *    L = E / R experts per rank, A alignment.  Logical rank r owns experts
 *    [r*L, (r+1)*L); ranks are partitions of one GPU buffer, not devices.
 *  - topk_idx is int64 [N, K] row-major; a negative entry is a masked slot;
 *    an entry >= E is an error (MOE_ERR_BAD_EXPERT_ID) and the slot is then
 *    treated as masked.
 *  - Slots and row indices are int32: N*K + E*(A-1) must be < 2^31.
 *  - Results are deterministic: the slot of a (token, k) pair inside its
 *    expert's segment is its rank in (token, k) order among that expert's
 *    pairs, independent of scheduling.  ([CS] §6.2/§6.4 hand out slots with
 *    atomics instead, so their order varies from run to run.)
 *  - Kernels are launched with programmatic dependent launch, and some of
 *    them start reading their inputs topk_idx, x and sf before the kernel in
 *    front of them on the stream has finished: the dispatch permutes prefetch
 *    token rows, the rank kernels stage ids.  This is safe after copies, after
 *    this library's own kernels (none of which writes those inputs) and after
 *    any kernel that does not release its dependents early.  The kernel
 *    launched on the stream directly before one of these calls must not write
 *    the call's topk_idx, x or sf and also release its dependents before it
 *    ends (griddepcontrol.launch_dependents /
 *    cudaTriggerProgrammaticLaunchCompletion): put an event record or any
 *    ordinary kernel between them.
 *
 * Kernels are compiled for sm_103a only.
 */
#ifndef MOE_LAYOUT_H_
#define MOE_LAYOUT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  0 is success. */
enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* host check failed: null pointer, bad size or alignment;
                                device (moe_dispatch_sf_col_major): map entry out of range */
  MOE_ERR_CUDA = 2,          /* a CUDA launch or copy failed                           */
  MOE_ERR_BAD_EXPERT_ID = 3, /* device: some topk_idx entry was >= E                   */
  MOE_ERR_CAPACITY = 4,      /* device: the layout needs more rows than capacity_rows  */
  MOE_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel ran out         */
  MOE_ERR_UNSUPPORTED = 6    /* host: sizes beyond what this build supports            */
};

/* Limits of this build.  Rows (token rows, scale rows, combine rows of
 * 2 * hidden bytes) longer than MOE_MAX_ROW_BYTES are refused with
 * MOE_ERR_UNSUPPORTED, which keeps every byte offset well inside int64. */
#define MOE_MAX_TOPK 32
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_ROW_BYTES (1 << 30)

/* Problem description.  Plain values, copied by every call. */
typedef struct moe_layout_desc {
  int64_t num_tokens;  /* N >= 0                                  */
  int32_t topk;        /* K, 1 <= K <= MOE_MAX_TOPK ([CS] §4.2)  */
  int32_t num_experts; /* E, 1 <= E <= MOE_MAX_EXPERTS           */
  int32_t num_ranks;   /* R >= 1, R divides E                     */
  int32_t alignment;   /* A >= 1 ([CS] §7.1-§7.2)                */
} moe_layout_desc;

/*
 * Bytes of device workspace the other calls need for this description
 * (sticky error word, grid-barrier words, the permute's work counter,
 * per-tile expert and rank histograms).  The workspace must
 * be zero-filled once before its first use (e.g. cudaMemsetAsync);
 * afterwards every call leaves it ready for the next.  One workspace serves
 * one stream at a time: calls that overlap on the GPU must not share it.
 * After MOE_ERR_TIMEOUT, zero-fill it again.
 */
MOE_API int moe_layout_workspace_bytes(const moe_layout_desc* desc, size_t* bytes);

/*
 * Count ([CS] §4.2).  Reads topk_idx [N*K]; writes
 *   expert_count[E]: number of (t, k) with topk_idx[t*K+k] == e;
 *   rank_count[R]:   number of tokens with at least one valid id in rank r,
 *                    each token counted once per rank (deduplicated);
 * and the per-tile histograms in `workspace` that moe_layout_scan needs.
 * Bad ids set MOE_ERR_BAD_EXPERT_ID in the workspace error word.
 */
MOE_API int moe_layout_count(const moe_layout_desc* desc, const int64_t* topk_idx,
                     int32_t* expert_count, int32_t* rank_count,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Prefix sums and slot maps ([CS] §5.2-§5.5, §7.2, §6.4).  Must follow
 * moe_layout_count on the same topk_idx, counts and workspace.  Writes
 *   expert_offset[E+1]: exclusive sum of align(expert_count[e], A); expert
 *                       e's segment is rows [expert_offset[e], expert_offset[e+1]);
 *                       rank r's block starts at expert_offset[r*L];
 *   rank_psum[R]:       inclusive sum of rank_count;
 *   dst_slot[N*K]:      row of (t, k) in the receive buffer, -1 if masked;
 *   src_idx[rows]:      token of each row, -1 for the alignment-gap rows;
 *   total_rows[1]:      expert_offset[E] (device scalar).
 * capacity_rows is the length of src_idx (and of the receive buffers).  If
 * the layout needs more rows, MOE_ERR_CAPACITY is recorded, src_idx is not
 * written and every dst_slot entry is -1.  A bound that never fails is
 * N*K + E*(A-1).
 */
MOE_API int moe_layout_scan(const moe_layout_desc* desc, const int64_t* topk_idx,
                    const int32_t* expert_count, const int32_t* rank_count,
                    void* workspace, size_t workspace_bytes,
                    int32_t* expert_offset, int32_t* rank_psum,
                    int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                    int32_t* total_rows, void* stream);

/*
 * moe_layout_count followed by moe_layout_scan, in one call, with the same
 * arguments and results.  For the largest batches (about a million pairs and
 * up), when every tile of the problem fits on the GPU at once, it runs as a
 * single cooperative kernel (count, per-expert scan over tiles, rank) with
 * two grid-wide barriers whose waits are bounded (MOE_ERR_TIMEOUT, after
 * which the workspace must be zero-filled again); otherwise it runs the two
 * calls' kernels.
 */
MOE_API int moe_layout_build(const moe_layout_desc* desc, const int64_t* topk_idx,
                             int32_t* expert_count, int32_t* rank_count,
                             void* workspace, size_t workspace_bytes,
                             int32_t* expert_offset, int32_t* rank_psum,
                             int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                             int32_t* total_rows, void* stream);

/*
 * moe_layout_build with int32 routing ids (topk_idx int32 [N*K]); same
 * results.  Frameworks that keep top-k ids as int32 avoid a widening copy.
 */
MOE_API int moe_layout_build_i32(const moe_layout_desc* desc, const int32_t* topk_idx,
                                 int32_t* expert_count, int32_t* rank_count,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* expert_offset, int32_t* rank_psum,
                                 int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                                 int32_t* total_rows, void* stream);

/*
 * Expand-mode dispatch permute ([CS] §6.3-§6.4, §8.2) with zero padding
 * ([CS] §7.3).  For every valid (t, k): recv_x row dst_slot[t*K+k] = x row t,
 * copied byte for byte (any row dtype: bf16, fp8, ...).  If sf is non-NULL
 * the scale-factor row sf[t] moves the same way into recv_sf.  With
 * zero_pad != 0, rows [expert_offset[e] + expert_count[e], expert_offset[e+1])
 * of recv_x (and recv_sf) are set to zero bytes.
 *   x [N, row_bytes], recv_x [capacity_rows, row_bytes]: row_bytes a positive
 *     multiple of 16, both base pointers 16-byte aligned;
 *   sf [N, sf_row_bytes], recv_sf [capacity_rows, sf_row_bytes]: sf_row_bytes
 *     a positive multiple of 4, pointers 4-byte aligned (NULL sf: no scale factors);
 *   dst_slot, expert_offset, expert_count: as written by the calls above.
 * Slots >= capacity_rows are not written and record MOE_ERR_CAPACITY.
 */
MOE_API int moe_dispatch_permute(const moe_layout_desc* desc, const void* x,
                         int64_t row_bytes, const void* sf, int64_t sf_row_bytes,
                         const int32_t* dst_slot, const int32_t* expert_offset,
                         const int32_t* expert_count, void* recv_x, void* recv_sf,
                         int64_t capacity_rows, int zero_pad, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Non-expand (rank-contiguous) slot map: the page's first scatter
 * ([CS] §6.2, §8.1-§8.2), where each token goes once to every logical rank
 * it reaches, whatever the number of that rank's experts it picked.  Must
 * follow moe_layout_build (or moe_layout_count + moe_layout_scan) on the same
 * topk_idx and workspace; rank_count is that call's output.  Writes
 *   rank_slot[N*K]: for each token and rank it reaches, the highest k among
 *                   the token's slots reaching that rank (the page's master
 *                   lane) gets the row index; every other slot gets -1;
 *   rank_src[rows]: token of each row.
 * Rank r's rows are [rank_psum[r] - rank_count[r], rank_psum[r]); tokens are
 * in ascending order inside it.  rows = rank_psum[R-1].  If rows exceed
 * capacity_rows, MOE_ERR_CAPACITY is recorded, every rank_slot is -1 and
 * rank_src is not written.  N*R rows always suffice.
 */
MOE_API int moe_layout_rank_rows(const moe_layout_desc* desc, const int64_t* topk_idx,
                                 const int32_t* rank_count, void* workspace, size_t workspace_bytes,
                                 int32_t* rank_slot, int32_t* rank_src, int64_t capacity_rows,
                                 void* stream);

/*
 * Non-expand dispatch permute ([CS] §6.3, §8.2 "non-expand"): recv row
 * rank_slot[t*K+k] = x row t for every slot that has a row; scale-factor
 * rows move alongside when sf is non-NULL.  No padding.  Argument rules as
 * for moe_dispatch_permute; rank_psum (from the layout) gives the row total
 * checked against capacity_rows.
 */
MOE_API int moe_dispatch_permute_ranks(const moe_layout_desc* desc, const void* x,
                                       int64_t row_bytes, const void* sf, int64_t sf_row_bytes,
                                       const int32_t* rank_slot, const int32_t* rank_psum,
                                       void* recv, void* recv_sf, int64_t capacity_rows,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scale factors of a receive buffer in column-major, TMA-aligned form.  The
 * page "00 DeepEP Engram Architecture Deep-Dive" (§1.1 Python API, §1.2 C++
 * runtime) names the option use_tma_aligned_col_major_sf and does not define
 * it.  Reading taken: the [rows, sf_cols] matrix of 4-byte scale words (fp32
 * scales, or packed exponents: moved verbatim) is stored column after
 * column, column j at recv_sf_cm + j*ld words, and ld is a multiple of 4 so
 * that every column starts on a 16-byte boundary (a TMA global stride must
 * be a multiple of 16 bytes).  Rows follow the layout's inverse map:
 *   recv_sf_cm[j*ld + i] = sf[src[i]*sf_cols + j]   for i < rows, src[i] >= 0;
 * rows with src[i] = -1 (the alignment gaps of the expand layout, [CS] §7.3)
 * are zero in every column when zero_pad != 0 and are not written
 * otherwise; rows >= rows are never written.
 *   sf [N, sf_cols] 4-byte words, 4-byte aligned; sf_cols >= 1;
 *   src: src_idx of moe_layout_build (expand layout) or rank_src of
 *        moe_layout_rank_rows (non-expand layout), entries in [-1, N);
 *   total_rows: device int32[1] holding rows: the total_rows output of
 *        moe_layout_build, or rank_psum + R - 1;
 *   recv_sf_cm [sf_cols, ld] words, 16-byte aligned, ld >= capacity_rows,
 *        ld a multiple of 4.
 * sf_cols above MOE_MAX_ROW_BYTES / 4 or ld above 2^32 return
 * MOE_ERR_UNSUPPORTED.
 * rows > capacity_rows records MOE_ERR_CAPACITY and nothing is written; a
 * src entry outside [-1, N) is skipped and records MOE_ERR_INVALID_ARG.
 * Independent of moe_dispatch_permute: call it instead of passing sf there,
 * on the same stream, after the layout.
 */
MOE_API int moe_dispatch_sf_col_major(const moe_layout_desc* desc, const void* sf, int64_t sf_cols,
                                      const int32_t* src, const int32_t* total_rows, void* recv_sf_cm,
                                      int64_t ld, int64_t capacity_rows, int zero_pad, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Combine: the inverse of the dispatch.  The pages keep the slot map for it
 * ([CS] §6.2) but print no arithmetic; this is the plain definition
 *   out[t, h] = bf16( sum over k = 0..K-1 with dst_slot[t*K+k] >= 0 of
 *                     weights[t*K+k] * float(expert_out[dst_slot[t*K+k], h]) )
 * accumulated in fp32 from 0 in ascending k with one fused multiply-add per
 * term, rounded once to bf16 (nearest, ties to even).  A token with no valid
 * slot gets zeros.
 *   expert_out bf16 [expert_out_rows, hidden]; out bf16 [N, hidden];
 *   weights fp32 [N*K]; hidden a positive multiple of 8; expert_out and out
 *   16-byte aligned.  Slots >= expert_out_rows are skipped and record
 *   MOE_ERR_CAPACITY.
 */
MOE_API int moe_combine_unpermute(const moe_layout_desc* desc, const void* expert_out,
                          int64_t expert_out_rows, int64_t hidden,
                          const int32_t* dst_slot, const float* weights,
                          void* out, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * moe_layout_build without a caller workspace, for callers that cannot
 * allocate device memory when they build the layout: for example an engine
 * that reserves all of HBM for its own allocator at start-up and forbids
 * cudaMalloc afterwards, a plugin that must not touch its host's memory
 * pool, or a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation.  The pages have no counterpart to this call; it
 * exists only for such callers.
 *
 * Inputs and outputs are the caller's, exactly as for moe_layout_build.  The
 * scratch is a fixed array of MOE_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 *  - Problems whose workspace (moe_layout_workspace_bytes) is larger than
 *    that are rejected with MOE_ERR_UNSUPPORTED before anything is launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it for that device's CUDA context; make
 *    that first call before any stream capture.  After a device reset the
 *    device has a new context and the array may sit at a new address: the
 *    first call in the new context looks it up again (again outside capture).
 *  - Every call on a device shares the array.  Each call clears the parts
 *    that must start at zero, but calls that overlap on the GPU (different
 *    streams, no ordering between them) race on it and give wrong results.
 *  - device_error: device int32 [1] that receives this call's device-side
 *    status (MOE_OK, MOE_ERR_BAD_EXPERT_ID, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT),
 *    written on `stream` after the layout.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
MOE_API int moe_layout_build_noalloc(const moe_layout_desc* desc, const int64_t* topk_idx,
                                     int32_t* expert_count, int32_t* rank_count,
                                     int32_t* expert_offset, int32_t* rank_psum,
                                     int32_t* dst_slot, int32_t* src_idx, int64_t capacity_rows,
                                     int32_t* total_rows, int32_t* device_error, void* stream);

/*
 * Running receive statistics ([CS] §7.2 keeps per-expert totals across
 * calls next to the alignment step): cumulative[e] += expert_count[e] for
 * every e, on `stream`, after a layout call.  cumulative is a caller-owned
 * device int64 [E] the caller zeroes once.
 */
MOE_API int moe_layout_accumulate_stats(const moe_layout_desc* desc, const int32_t* expert_count,
                                        int64_t* cumulative, void* stream);

/*
 * Dispatch straight from host memory: the ids (and, if given, the top-k
 * weights and fp8 scale factors) are copied to the caller's device staging
 * buffers, the layout is built (moe_layout_build), and the token rows are
 * copied in chunks of chunk_tokens tokens (0 = one chunk) on copy_stream
 * while the permute (moe_dispatch_permute, zero padding on the first chunk)
 * of each chunk runs on `stream` as soon as its rows have landed.  Results
 * and errors are those of the two calls; on return everything is enqueued
 * on `stream` (copy_stream is joined into it).  Host buffers must be
 * page-locked for the copies to overlap.  A pipeline around the method's
 * steps; the pages have no counterpart to it.
 *   topk_idx_host [N*K] int64, x_host [N, row_bytes], sf_host [N, sf_row_bytes]
 *   or NULL, weights_host [N*K] fp32 or NULL (with weights NULL too);
 *   topk_idx, x, sf, weights: device buffers of the same sizes.
 */
MOE_API int moe_dispatch_from_host(const moe_layout_desc* desc, const int64_t* topk_idx_host,
                                   const void* x_host, int64_t row_bytes, const void* sf_host,
                                   int64_t sf_row_bytes, const float* weights_host,
                                   int64_t* topk_idx, void* x, void* sf, float* weights,
                                   int32_t* expert_count, int32_t* rank_count,
                                   int32_t* expert_offset, int32_t* rank_psum,
                                   int32_t* dst_slot, int32_t* src_idx, int32_t* total_rows,
                                   void* recv_x, void* recv_sf, int64_t capacity_rows,
                                   void* workspace, size_t workspace_bytes,
                                   int64_t chunk_tokens, void* stream, void* copy_stream);

/*
 * Combine straight to host memory: moe_combine_unpermute runs in chunks of
 * chunk_tokens tokens (0 = one chunk) on `stream` into the device buffer
 * `out` [N, hidden] bf16, and each chunk is copied to out_host on
 * copy_stream while the next chunk is combined; copy_stream is joined into
 * `stream` at the end, so synchronising `stream` covers the copies.
 * out_host must be page-locked for the copies to overlap.  A pipeline
 * around the method's steps; the pages have no counterpart to it.
 */
MOE_API int moe_combine_to_host(const moe_layout_desc* desc, const void* expert_out,
                                int64_t expert_out_rows, int64_t hidden,
                                const int32_t* dst_slot, const float* weights, void* out,
                                void* out_host, void* workspace, size_t workspace_bytes,
                                int64_t chunk_tokens, void* stream, void* copy_stream);

/*
 * Synchronise `stream`, copy the workspace's sticky error word (the first
 * device-side error since the last read; MOE_OK if none) into
 * *device_error, and reset it to MOE_OK.
 */
MOE_API int moe_layout_get_error(void* workspace, int32_t* device_error, void* stream);

/* Static, human-readable name of a status code. */
MOE_API const char* moe_strerror(int status);

/* Number of kernels this library has launched in this process so far. */
MOE_API uint64_t moe_kernel_launches(void);

/*
 * Test hook for the bounded waits (not for normal use; process-wide; affects
 * launches made after the call).  Every wait inside the library's kernels
 * gives up after limit_ns nanoseconds (0: the default, 1 s; at most 1 s),
 * records MOE_ERR_TIMEOUT and lets the kernel finish.  barrier_extra > 0
 * raises the cooperative layout kernel's grid-barrier targets past the number
 * of CTAs, so its first barrier can only run out; extra_tx (a multiple of 16)
 * adds transaction bytes that no copy delivers to each CTA's first stage of
 * the dynamic permute, so that stage can only run out.  A layout that timed
 * out leaves its workspace's barrier counter set: zero the workspace before
 * reusing it.  Call with (0, 0, 0) to restore normal operation.
 */
MOE_API int moe_debug_set_waits(uint64_t limit_ns, uint32_t barrier_extra, uint32_t extra_tx);

/*
 * The CUDA error code (cudaError_t) behind this thread's most recent
 * MOE_ERR_CUDA from any entry point, or 0 if there was none; *message (if
 * non-NULL) receives its description.  Diagnostics only: a status the pages
 * do not define.
 */
MOE_API int moe_last_cuda_error(const char** message);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYOUT_H_ */
