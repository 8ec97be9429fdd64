/*
 * CPU oracle for the DCP top-K merge (test infrastructure only; see
 * dcp_topk_oracle.c).  All pointers are host memory.  Returns 0 on success,
 * 1 on invalid arguments, 2 on allocation failure.
 */
#ifndef DCP_TOPK_ORACLE_H
#define DCP_TOPK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Rank-major candidates scores/ids (dcp, T, K); outputs (T, K) row-major. */
int oracle_merge(const float* scores, const int32_t* ids, int T, int dcp, int K,
                 const int32_t* row_starts, int32_t* out_ids, float* out_scores);

/* Same, for the listed rows only (rows[i] in [0, T)); outputs (nrows, K). */
int oracle_merge_rows(const float* scores, const int32_t* ids, int T, int dcp, int K,
                      const int32_t* row_starts, const int32_t* rows, int nrows,
                      int32_t* out_ids, float* out_scores);

/* One rank's local top-K over logits rows (T, ld), first L columns used. */
int oracle_local_topk(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                      const int32_t* row_starts, float* out_scores, int32_t* out_ids);

/* Top-K over all shards' logits (dcp, T, ld) at once, ids r*L + c. */
int oracle_fused_topk(const float* logits, int T, int dcp, int L, int ld, int K,
                      const int32_t* row_starts, float* out_scores, int32_t* out_ids);

/* The same two with the shard id layout chosen: interleaved = 0 gives ids
 * r*L + c (contiguous shards), interleaved = 1 gives ids c*dcp + r. */
int oracle_local_topk_ids(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                          const int32_t* row_starts, int interleaved, float* out_scores,
                          int32_t* out_ids);
int oracle_fused_topk_ids(const float* logits, int T, int dcp, int L, int ld, int K,
                          const int32_t* row_starts, int interleaved, float* out_scores,
                          int32_t* out_ids);

#ifdef __cplusplus
}
#endif

#endif
