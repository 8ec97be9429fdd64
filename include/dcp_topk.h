/*
 * dcp_topk.h -- C ABI of the GB300 (sm_103a) DCP sparse-indexer top-K library.
 *
 * Decode context parallelism (DCP) shards the KV cache across `dcp` ranks.
 * Each rank keeps the top-K of its own shard's indexer logits; the merge then
 * picks, per query row, the global top-K of the dcp*K gathered candidates
 * ("[Kernel] Optimize CuTeDSL DCP top-k merge", Summary).  Here every shard
 * lives in one GPU's memory, so no collective is involved.
 *
 * Selection order (all entry points): score descending, then lowest global
 * token id; equivalently the 64-bit key (score_key(s) << 32) | ~id taken as
 * unsigned, where score_key is the order-preserving map of the fp32 bits to
 * u32 and ~id is the bitwise complement of the id as unsigned 32-bit
 * ("[Kernel] Optimize CuTeDSL DCP top-k merge", Summary).  Consequences:
 * +0.0 ranks above -0.0; among equal scores the smallest unsigned id wins,
 * so a padding slot (score -inf, id -1) ranks below every real candidate.
 * Output rows list the K winners in that order; scores are copied bit for bit.
 * Results are deterministic: identical inputs give identical output bits.
 * NaN scores are outside the contract.
 *
 * Conventions for every entry point:
 *  - all data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no pointer after the call returns;
 *  - work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call does not synchronise, so results are ready only
 *    when the stream reaches that point; calls issue no host-device sync and
 *    may be captured in a CUDA graph once the device has been used by a
 *    first (uncaptured) call of the same entry point;
 *  - kernels are launched with programmatic stream serialization: one may be
 *    scheduled while the stream's previous kernel drains, but it waits for
 *    that kernel to complete (its writes visible) before touching memory, so
 *    stream order is unchanged;
 *  - outputs must not overlap inputs;
 *  - argument errors are reported before anything is enqueued.
 */
#ifndef DCP_TOPK_H
#define DCP_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dcp_stream_t; /* same type as cudaStream_t */

typedef enum {
    DCP_OK = 0,
    DCP_ERR_INVALID = 1,     /* a null required pointer or an out-of-range size */
    DCP_ERR_UNSUPPORTED = 2, /* valid, but beyond this build's limits (the caller may fall back) */
    DCP_ERR_CUDA = 3         /* a CUDA runtime error while preparing or launching */
} dcp_status;

/* Compiled limits: K <= DCP_MAX_K, candidates per row (dcp*K, or L for the
 * local top-K, or dcp*L for the fused top-K) <= DCP_MAX_CANDIDATES. */
#define DCP_MAX_K 4096
#define DCP_MAX_CANDIDATES 16384

/*
 * dcp_topk_merge -- global top-K of per-shard candidates.
 *
 * The merge of "[Kernel] Optimize CuTeDSL DCP top-k merge" (Summary), reading
 * the gathered candidates in the rank-major layout of "Reserve the sparse
 * indexer's DCP top-k merge scratch through the workspace manager" (Purpose)
 * directly, without moving the rank dimension inside first.
 *
 *   scores      fp32 [dcp][T][K], rank-major: shard r's candidates for row t
 *               start at scores + (r*T + t)*K.
 *   ids         int32 [dcp][T][K], same layout; -1 marks a padding slot.
 *   T, dcp, K   rows, shards, candidates per shard (= outputs per row).
 *               T == 0 is a no-op returning DCP_OK.
 *   row_starts  int32 [T] or NULL (all zero): added to every output id that is
 *               not -1, per row (the per-row offsets of the second page,
 *               Purpose).  The caller keeps id + row_starts[t] within int32.
 *   out_ids     int32 [T][K] row-major.
 *   out_scores  fp32  [T][K] row-major.
 *   workspace   may be NULL: this build needs no scratch
 *               (dcp_topk_merge_workspace_size reports 0 bytes).
 *
 * Errors: DCP_ERR_INVALID for T < 0, dcp < 1, K < 1, or a NULL scores, ids,
 * out_ids or out_scores with T > 0; DCP_ERR_UNSUPPORTED for K > DCP_MAX_K,
 * dcp*K > DCP_MAX_CANDIDATES, or a workspace smaller than the reported size;
 * DCP_ERR_CUDA if the launch fails.
 *
 * Rows are independent; the rows are processed in chunks of 1024 by a
 * persistent grid ("Reserve the sparse indexer's DCP top-k merge scratch
 * through the workspace manager", Purpose), and the result does not depend
 * on the chunking.
 *
 * On-chip resources: with K = 2048, dcp <= 4 and more than two rows per SM
 * the kernel holds 64 tensor-memory columns per CTA (four CTAs, 256 of an
 * SM's 512 columns) while it runs.  Its allocation waits in hardware for free
 * columns, so a kernel on another stream that holds tensor memory on the same
 * SM can delay it (and be delayed by it); neither waits on the other.
 */
dcp_status dcp_topk_merge(const float* scores, const int32_t* ids, int T, int dcp, int K,
                          const int32_t* row_starts, int32_t* out_ids, float* out_scores,
                          void* workspace, size_t workspace_bytes, dcp_stream_t stream);

/*
 * dcp_topk_merge_shards -- dcp_topk_merge over shards that live in separate
 * allocations, read where they lie.
 *
 * "[DCP][Performance] Add Shared-DCP peer-addressable decode data paths"
 * (Summary; Top-K performance) has the Top-K consumer read owner-local and
 * peer shards through views instead of first gathering them into one inbox.
 * On one GPU that is a merge whose shards are separate buffers: the same
 * selection and order as dcp_topk_merge, without the copy that would stack
 * them into a rank-major (dcp, T, K) buffer.
 *
 *   shard_scores  DEVICE array of dcp pointers; shard_scores[r] points to
 *                 fp32 [T][K] row-major: shard r's candidates for row t
 *                 start at shard_scores[r] + t*K.
 *   shard_ids     DEVICE array of dcp pointers to int32 [T][K] the same way;
 *                 -1 marks a padding slot.
 *   T, dcp, K, row_starts, out_ids, out_scores   as dcp_topk_merge.
 *
 * The two pointer arrays are read on the device during the launch, so they
 * (and the shards) must stay valid and unchanged until the stream passes the
 * call; a captured CUDA graph reads them again at each replay, so a caller
 * may repoint shards between replays by rewriting the arrays.  When K is a
 * multiple of 4 every shard pointer must be 16-byte aligned: the kernels
 * check this on the device and, if it fails, set
 * DCP_DEVICE_BAD_SHARD_ALIGNMENT in the device status word
 * (dcp_topk_device_status) and fill the affected rows with id
 * DCP_ID_UNWRITTEN and NaN scores instead of reading them.
 *
 * Errors: DCP_ERR_INVALID for T < 0, dcp < 1, K < 1, a NULL array or output
 * with T > 0, or a pointer array the device cannot read (host-only memory);
 * DCP_ERR_UNSUPPORTED for K > DCP_MAX_K or dcp*K > DCP_MAX_CANDIDATES;
 * DCP_ERR_CUDA if the launch fails.  No workspace: nothing is staged.
 */
dcp_status dcp_topk_merge_shards(const float* const* shard_scores, const int32_t* const* shard_ids,
                                 int T, int dcp, int K, const int32_t* row_starts,
                                 int32_t* out_ids, float* out_scores, dcp_stream_t stream);

/*
 * dcp_topk_merge_workspace_size -- scratch bytes dcp_topk_merge needs for
 * these sizes (the merge reserved its scratch through a workspace manager in
 * "Reserve the sparse indexer's DCP top-k merge scratch through the workspace
 * manager", Purpose).  Writes 0: this build keeps every intermediate on chip.
 * Errors as dcp_topk_merge's size checks; `bytes` must not be NULL.
 */
dcp_status dcp_topk_merge_workspace_size(int T, int dcp, int K, size_t* bytes);

/*
 * dcp_local_topk -- one rank's top-K over its own shard of indexer logits,
 * the per-rank step before the merge ("[Kernel] Optimize CuTeDSL DCP top-k
 * merge", Summary: each rank holds the local top-K of its 1/DCP KV shard).
 *
 *   logits      fp32 [T][ld], row-major; the first L columns of a row are this
 *               rank's L local KV positions.
 *   T, L, ld    rows, local columns, row stride in elements (ld >= L).
 *   K           outputs per row; if L < K the row is padded with (-inf, -1).
 *   rank, dcp   this rank and the number of shards (0 <= rank < dcp).
 *   row_starts  int32 [T] or NULL (all zero).
 *   out_scores  fp32  [T][K] row-major: this rank's slice of the rank-major
 *               candidate buffer dcp_topk_merge reads (scores + rank*T*K).
 *   out_ids     int32 [T][K]: global ids row_starts[t] + rank*L + column.
 *
 * Contiguous shards are this library's reading of the global id (the pages do
 * not fix it): shard r owns local positions [r*L, (r+1)*L).  row_starts should
 * be given to either this call or the merge, not both.
 *
 * Errors: DCP_ERR_INVALID for T < 0, L < 1, ld < L, K < 1, dcp < 1, rank out of
 * range, or a NULL logits/out pointer with T > 0; DCP_ERR_UNSUPPORTED for
 * K > DCP_MAX_K or L > DCP_MAX_CANDIDATES; DCP_ERR_CUDA if the launch fails.
 */
dcp_status dcp_local_topk(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                          const int32_t* row_starts, float* out_scores, int32_t* out_ids,
                          dcp_stream_t stream);

/*
 * dcp_fused_topk -- the local top-K of every shard and their merge in one
 * pass: the global top-K over all dcp*L logits of each row.  Each rank keeps
 * the local top-K of its shard and the merge picks the global top-K of those
 * ("[Kernel] Optimize CuTeDSL DCP top-k merge", Summary); every global winner
 * is among its shard's local top-K, so selecting straight from the logits
 * gives the same result as dcp_local_topk on every shard followed by
 * dcp_topk_merge, without the candidate round trip through memory.
 *
 *   logits      fp32 [dcp][T][ld], rank-major: shard r's row t starts at
 *               logits + (r*T + t)*ld; its first L columns are candidates.
 *   T, dcp      rows and shards.  T == 0 is a no-op returning DCP_OK.
 *   L, ld       columns per shard and row stride in elements (ld >= L).
 *   K           outputs per row; rows with dcp*L < K are padded (-inf, -1).
 *   row_starts  int32 [T] or NULL (all zero).
 *   out_scores  fp32  [T][K] row-major, sorted as for the merge.
 *   out_ids     int32 [T][K]: global ids row_starts[t] + r*L + column.
 *
 * Errors: DCP_ERR_INVALID for T < 0, dcp < 1, L < 1, ld < L, K < 1, or a NULL
 * logits/out pointer with T > 0; DCP_ERR_UNSUPPORTED for K > DCP_MAX_K or
 * dcp*L > DCP_MAX_CANDIDATES; DCP_ERR_CUDA if the launch fails.
 */
dcp_status dcp_fused_topk(const float* logits, int T, int dcp, int L, int ld, int K,
                          const int32_t* row_starts, float* out_scores, int32_t* out_ids,
                          dcp_stream_t stream);

/*
 * Shard id layouts for the local and fused top-K.  The pages do not fix how a
 * rank's local KV positions map to global token ids:
 *   DCP_IDS_CONTIGUOUS   column c of rank r is id r*L + c (shard r owns
 *                        [r*L, (r+1)*L)); what dcp_local_topk and
 *                        dcp_fused_topk use.
 *   DCP_IDS_INTERLEAVED  column c of rank r is id c*dcp + r (tokens dealt to
 *                        the ranks round-robin).
 * In both the id grows with the column within a shard, so the local top-K of
 * every shard followed by dcp_topk_merge still equals the fused top-K.
 */
typedef enum { DCP_IDS_CONTIGUOUS = 0, DCP_IDS_INTERLEAVED = 1 } dcp_id_layout;

/*
 * dcp_local_topk_ex -- dcp_local_topk with the shard id layout chosen:
 * out_ids are row_starts[t] + rank*L + column (DCP_IDS_CONTIGUOUS) or
 * row_starts[t] + column*dcp + rank (DCP_IDS_INTERLEAVED).  Among equal
 * scores the lower id ranks first.  Other arguments and errors as
 * dcp_local_topk; a layout outside the enum is DCP_ERR_INVALID.
 */
dcp_status dcp_local_topk_ex(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                             const int32_t* row_starts, int layout, float* out_scores,
                             int32_t* out_ids, dcp_stream_t stream);

/*
 * dcp_fused_topk_ex -- dcp_fused_topk with the shard id layout chosen: ids are
 * row_starts[t] + r*L + column or row_starts[t] + column*dcp + r, and among
 * equal scores the lower id ranks first.  Other arguments and errors as
 * dcp_fused_topk; a layout outside the enum is DCP_ERR_INVALID.
 */
dcp_status dcp_fused_topk_ex(const float* logits, int T, int dcp, int L, int ld, int K,
                             const int32_t* row_starts, int layout, float* out_scores,
                             int32_t* out_ids, dcp_stream_t stream);

/*
 * dcp_topk_device_status -- reads and clears the device-side status word of
 * the current device.  Kernels that stage rows with bulk copies wait for each
 * copy with a bounded poll (about a second); if a copy never lands, the
 * kernel sets DCP_DEVICE_COPY_TIMEOUT here and that CTA stops.  The call that
 * launched it has already returned DCP_OK, so the status word is the only
 * report.  The rows that CTA had not finished (its current row and the rows
 * it would still have walked) are filled with id DCP_ID_UNWRITTEN and a NaN
 * score; the rest of the call's output is valid.  Before stopping, the CTA
 * gives its copies one more bounded wait; a copy that still has not landed
 * may complete into that CTA's (released) shared memory afterwards, so no
 * wait anywhere is unbounded.  0 means no failure since the last read.
 *
 *   status  host pointer receiving the word (DCP_ERR_INVALID if NULL).
 *
 * Synchronises the device first (cudaDeviceSynchronize), so call it outside
 * any stream capture.  DCP_ERR_CUDA on a CUDA error.  This diagnostic has no
 * counterpart on the pages; it is how a bounded wait reports that it gave up.
 */
#define DCP_DEVICE_COPY_TIMEOUT 1u
#define DCP_DEVICE_BAD_SHARD_ALIGNMENT 2u /* a separate shard not 16-byte aligned */
#define DCP_ID_UNWRITTEN INT32_MIN /* id of an output slot a kernel could not fill */
dcp_status dcp_topk_device_status(unsigned int* status);

/*
 * dcp_topk_selftest_wait_timeout -- launches, on `stream`, one CTA that arms
 * a copy barrier for a copy it never issues and waits for it for at most
 * `wait_cycles` SM clock cycles, so that the timeout path runs: the next
 * dcp_topk_device_status then reports DCP_DEVICE_COPY_TIMEOUT.  For tests;
 * no counterpart on the pages.  DCP_ERR_CUDA if the launch fails.
 */
dcp_status dcp_topk_selftest_wait_timeout(unsigned int wait_cycles, dcp_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* dcp_status_string(dcp_status status);

#ifdef __cplusplus
}
#endif

#endif /* DCP_TOPK_H */
