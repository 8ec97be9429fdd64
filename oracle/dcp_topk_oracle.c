/*
 * CPU oracle for the DCP sparse-indexer top-K merge and the per-shard local
 * top-K.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the bench's
 * CPU-baseline leg call it; the product path never does.  It shares no code,
 * header or constant with the CUDA library.
 *
 * Plain, single-threaded, obviously-correct C: for every query row it gathers
 * the row's candidates, sorts them with the C library's qsort under the 64-bit
 * key the selector is defined by, and keeps the first K.  There is no blocking,
 * fusion or reordering beyond that definition.
 *
 * Sources (vLLM pull-request pages):
 *  - "[Kernel] Optimize CuTeDSL DCP top-k merge", Summary: each rank holds the
 *    local top-K of its 1/DCP KV shard, the merge selects the global top-K of
 *    the gathered candidates; the reference order is the 64-bit key
 *    score<<32 | ~id, i.e. score descending, then lowest global token id;
 *    selection is deterministic.
 *  - "Reserve the sparse indexer's DCP top-k merge scratch through the
 *    workspace manager", Purpose: candidates are gathered rank-major,
 *    (dcp*T, K); row_starts are applied per row; rows are independent, so
 *    chunking the rows does not change the result.
 *
 * Readings where the pages leave a step open (each is pinned by a test):
 *  - score key: the order-preserving map of fp32 bits to u32 (negative floats
 *    bit-inverted, non-negative floats with the sign bit set), so -0.0 ranks
 *    below +0.0 and -inf lowest;
 *  - ~id is taken as unsigned 32-bit, so among equal scores the lowest
 *    unsigned id wins and padding (id -1) ranks last;
 *  - the output is the K winners in key order, scores copied bit for bit;
 *  - row_starts[t] (0 when absent) is added to every non-padding output id of
 *    the merge, and to every id the local top-K emits;
 *  - local top-K ids are row_starts[t] + rank*L + column (contiguous shards,
 *    the default) or row_starts[t] + column*dcp + rank (interleaved shards),
 *    and rows with fewer than K columns are padded with (-inf, -1).
 *
 * Parity is pinned for every exported function (hand-worked examples, brute
 * force on tiny inputs, invariants, the local/merge composition identity).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "dcp_topk_oracle.h"

/* Order-preserving fp32 -> u32 score key (the "32-bit score key"). */
static uint32_t score_key(float s)
{
    uint32_t b;
    memcpy(&b, &s, sizeof b);
    if (b & 0x80000000u)
        return ~b;
    return b | 0x80000000u;
}

/* The 64-bit selection key: score key in the high word, inverted id below. */
static uint64_t cand_key(float s, uint32_t id)
{
    return ((uint64_t)score_key(s) << 32) | (uint64_t)(uint32_t)(~id);
}

typedef struct {
    uint64_t key;
    int64_t pos; /* gather position, a stable tie-break for identical keys */
    float score;
    int32_t id;
} cand_t;

static int by_key_desc(const void* pa, const void* pb)
{
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->key != b->key)
        return a->key > b->key ? -1 : 1;
    if (a->pos != b->pos)
        return a->pos < b->pos ? -1 : 1;
    return 0;
}

static void merge_one_row(const float* scores, const int32_t* ids, int T, int dcp, int K,
                          int t, int32_t row_start, cand_t* buf,
                          int32_t* out_ids, float* out_scores)
{
    int64_t n = 0;
    /* Gather in rank-major order: shard r's K candidates of row t. */
    for (int r = 0; r < dcp; ++r) {
        const int64_t base = ((int64_t)r * T + t) * (int64_t)K;
        for (int k = 0; k < K; ++k) {
            buf[n].score = scores[base + k];
            buf[n].id = ids[base + k];
            buf[n].key = cand_key(buf[n].score, (uint32_t)buf[n].id);
            buf[n].pos = n;
            ++n;
        }
    }
    qsort(buf, (size_t)n, sizeof(cand_t), by_key_desc);
    for (int j = 0; j < K; ++j) {
        out_scores[j] = buf[j].score;
        out_ids[j] = buf[j].id == -1 ? -1 : (int32_t)((uint32_t)buf[j].id + (uint32_t)row_start);
    }
}

int oracle_merge_rows(const float* scores, const int32_t* ids, int T, int dcp, int K,
                      const int32_t* row_starts, const int32_t* rows, int nrows,
                      int32_t* out_ids, float* out_scores)
{
    if (T < 0 || dcp < 1 || K < 1 || nrows < 0)
        return 1;
    if (nrows == 0)
        return 0;
    cand_t* buf = (cand_t*)malloc(sizeof(cand_t) * (size_t)dcp * (size_t)K);
    if (!buf)
        return 2;
    for (int i = 0; i < nrows; ++i) {
        const int t = rows ? rows[i] : i;
        if (t < 0 || t >= T) {
            free(buf);
            return 1;
        }
        merge_one_row(scores, ids, T, dcp, K, t, row_starts ? row_starts[t] : 0, buf,
                      out_ids + (int64_t)i * K, out_scores + (int64_t)i * K);
    }
    free(buf);
    return 0;
}

int oracle_merge(const float* scores, const int32_t* ids, int T, int dcp, int K,
                 const int32_t* row_starts, int32_t* out_ids, float* out_scores)
{
    return oracle_merge_rows(scores, ids, T, dcp, K, row_starts, NULL, T, out_ids, out_scores);
}

/* Global id (before row_starts) of column c of rank r's shard: contiguous
 * shards own [r*L, (r+1)*L); interleaved shards own the ids = r (mod dcp),
 * column c being id c*dcp + r. */
static uint32_t shard_id(int interleaved, int r, int dcp, int L, int c)
{
    if (interleaved)
        return (uint32_t)c * (uint32_t)dcp + (uint32_t)r;
    return (uint32_t)r * (uint32_t)L + (uint32_t)c;
}

int oracle_local_topk_ids(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                          const int32_t* row_starts, int interleaved, float* out_scores,
                          int32_t* out_ids)
{
    /* Rank `rank`'s top-K over its L columns, ordered by (score, global id). */
    if (T < 0 || L < 1 || ld < L || K < 1 || dcp < 1 || rank < 0 || rank >= dcp ||
        (interleaved != 0 && interleaved != 1))
        return 1;
    if (T == 0)
        return 0;
    cand_t* buf = (cand_t*)malloc(sizeof(cand_t) * (size_t)L);
    if (!buf)
        return 2;
    for (int t = 0; t < T; ++t) {
        const float* row = logits + (int64_t)t * ld;
        for (int c = 0; c < L; ++c) {
            const uint32_t gid = shard_id(interleaved, rank, dcp, L, c);
            buf[c].score = row[c];
            buf[c].id = (int32_t)gid;
            buf[c].key = cand_key(row[c], gid);
            buf[c].pos = c;
        }
        qsort(buf, (size_t)L, sizeof(cand_t), by_key_desc);
        const uint32_t base = row_starts ? (uint32_t)row_starts[t] : 0u;
        for (int j = 0; j < K; ++j) {
            if (j < L) {
                out_scores[(int64_t)t * K + j] = buf[j].score;
                out_ids[(int64_t)t * K + j] = (int32_t)(base + (uint32_t)buf[j].id);
            } else {
                out_scores[(int64_t)t * K + j] = -INFINITY;
                out_ids[(int64_t)t * K + j] = -1;
            }
        }
    }
    free(buf);
    return 0;
}

int oracle_local_topk(const float* logits, int T, int L, int ld, int K, int rank, int dcp,
                      const int32_t* row_starts, float* out_scores, int32_t* out_ids)
{
    return oracle_local_topk_ids(logits, T, L, ld, K, rank, dcp, row_starts, 0, out_scores,
                                 out_ids);
}

int oracle_fused_topk_ids(const float* logits, int T, int dcp, int L, int ld, int K,
                          const int32_t* row_starts, int interleaved, float* out_scores,
                          int32_t* out_ids)
{
    /* Top-K taken directly over all dcp*L logits of a row, global id
     * row_starts[t] + shard_id(r, c): the result the local top-K followed by
     * the merge must reproduce. */
    if (T < 0 || dcp < 1 || L < 1 || ld < L || K < 1 || (interleaved != 0 && interleaved != 1))
        return 1;
    if (T == 0)
        return 0;
    const int64_t n = (int64_t)dcp * L;
    cand_t* buf = (cand_t*)malloc(sizeof(cand_t) * (size_t)n);
    if (!buf)
        return 2;
    for (int t = 0; t < T; ++t) {
        int64_t m = 0;
        for (int r = 0; r < dcp; ++r) {
            const float* row = logits + ((int64_t)r * T + t) * ld;
            for (int c = 0; c < L; ++c) {
                const uint32_t gid = shard_id(interleaved, r, dcp, L, c);
                buf[m].score = row[c];
                buf[m].id = (int32_t)gid;
                buf[m].key = cand_key(row[c], gid);
                buf[m].pos = m;
                ++m;
            }
        }
        qsort(buf, (size_t)n, sizeof(cand_t), by_key_desc);
        const uint32_t base = row_starts ? (uint32_t)row_starts[t] : 0u;
        for (int j = 0; j < K; ++j) {
            if (j < n) {
                out_scores[(int64_t)t * K + j] = buf[j].score;
                out_ids[(int64_t)t * K + j] = (int32_t)(base + (uint32_t)buf[j].id);
            } else {
                out_scores[(int64_t)t * K + j] = -INFINITY;
                out_ids[(int64_t)t * K + j] = -1;
            }
        }
    }
    free(buf);
    return 0;
}

int oracle_fused_topk(const float* logits, int T, int dcp, int L, int ld, int K,
                      const int32_t* row_starts, float* out_scores, int32_t* out_ids)
{
    return oracle_fused_topk_ids(logits, T, dcp, L, ld, K, row_starts, 0, out_scores, out_ids);
}
