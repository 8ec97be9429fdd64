// topk_fast.cuh -- the streaming top-K path for rows of up to 8192 candidates
// and K <= 2048 (the merge at DCP=4, K=2048 and the local top-K over 4096
// columns fall here).
//
// A persistent grid of one 1024-thread CTA per SM walks the rows; each CTA
// double-buffers its rows in shared memory with 16-byte cp.async copies, so
// the next row streams in from HBM while the current one is selected.  The
// selection and the final ordering come out of one two-level bucket pass
// instead of a radix select followed by a sort:
//
//  L1  an 11-bit histogram of the score key's top bits over every candidate
//      (the "radix pass over 32-bit score keys first" of "[Kernel] Optimize
//      CuTeDSL DCP top-k merge", Summary) locates the bin b1 that holds the
//      K-th largest key; every candidate above b1 is a winner.
//  L2  bins >= b1 are split into fine buckets, about one bucket per two
//      candidates, on the next bits of the candidate's 64-bit key
//      score_key<<32 | ~id below the bin prefix, skipping bits constant over
//      the row; the token id therefore only enters when scores tie, which is
//      the page's conditional tie-break.  Fine buckets are ordered like the
//      keys, so a prefix sum over their counts gives each bucket its first
//      output position.
//  RANK each candidate in a bucket that starts before K counts the bucket
//      members with a larger key; bucket start + that count is its output
//      position, and positions >= K are the losers.  Buckets are small (a few
//      members), so this is both the selection of the threshold and the sort.
//
// Rows whose buckets come out too large to rank this way (pathological key
// clusters) take the radix-select + sort path of topk_core.cuh on the same
// staged row, so results never depend on the data's distribution, only the
// speed does.
//
// Barriers: every shared array is reset only after the barrier that follows
// its last reader in the row (the race the first page's review reports came
// from resetting shared state that late warps had not yet read).
#pragma once

#include <cstdint>

#include "topk_core.cuh"

namespace dcp {

constexpr int kFastItems = 8;
constexpr int kFastMaxN = kThreads * kFastItems;  // 8192 candidates per row
constexpr int kFastMaxK = 2048;
constexpr int kFineMax = kFastMaxK + 1024;        // fine buckets per row, upper bound
constexpr int kArrSlack = 256;                    // room for the bucket straddling K
constexpr int kArrMax = kFastMaxK + kArrSlack;
constexpr uint32_t kRankLimit = 1u << 19;         // sum of squared bucket sizes
constexpr uint32_t kNoBucket = 0xFFFFFFFFu;

struct FastShared {
  SelectShared sel;                 // radix-select state of the fallback path
  uint32_t table[kHistBins];        // L1 counts, then per bin (first bucket << 8 | log2 buckets)
  uint32_t fcnt[kFineMax];          // L2 counts (+ 1<<16 per member of an exact bucket), then cursors
  uint32_t fst[kFineMax];           // bucket start | count << 15 | exact << 31
  unsigned long long arr[kArrMax];  // candidates in bucket order (fallback: sorted winners)
  uint32_t out_s[kFastMaxK];        // winners' score bits in output order
  int32_t out_i[kFastMaxK];         // winners' output ids
  uint32_t wa[kWarps];
  uint32_t wb[kWarps];
  // OR / AND over the candidates of each key class (0: positive scores,
  // 1: negative finite scores, 2: -inf and below) of the low 21 key bits
  // (entries 0..2) and of the inverted ids (entries 3..5)
  uint32_t acc_or[6];
  uint32_t acc_and[6];
  uint32_t b1;                      // bin of the K-th largest key
  uint32_t nfine;                   // buckets in bins >= b1
  uint32_t rank_work;               // sum of squared sizes of the buckets to rank
  uint32_t arr_overflow;            // a bucket straddling K would not fit arr
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Buckets given to an L1 bin holding h candidates: half of h rounded up to a
// power of two, at least 1 and at most 1024; 0 for an empty bin.
__device__ __forceinline__ uint32_t fine_buckets(uint32_t h) {
  if (h == 0u) return 0u;
  if (h <= 2u) return 1u;
  const uint32_t p = 1u << (32 - __clz(h - 1u));  // next power of two >= h
  return min(p >> 1, 1024u);
}

// Key class of a score key: 0 for positive scores, 1 for negative finite
// scores, 2 for -inf and below (L1 bins 0..3), where padding lives.
__device__ __forceinline__ int key_class(uint32_t k) {
  return (k & 0x80000000u) ? 0 : ((k >> 21) <= 3u ? 2 : 1);
}

template <class Source>
__global__ void __launch_bounds__(kThreads, 1)
    topk_fast_kernel(Source src, int T, int K, float* __restrict__ out_scores,
                     int32_t* __restrict__ out_ids) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FastShared& s = *reinterpret_cast<FastShared*>(smem_raw);
  const int n = src.count();
  const int words = (src.staged_words() + 3) & ~3;
  uint32_t* rowbuf = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(FastShared) + 15) & ~(size_t)15));
  const int ksel = K < n ? K : n;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < kHistBins; i += kThreads) s.table[i] = 0u;
  for (int i = tid; i < kFineMax; i += kThreads) s.fcnt[i] = 0u;
  if (tid < 6) {
    s.acc_or[tid] = 0u;
    s.acc_and[tid] = 0xFFFFFFFFu;
  }
  if (tid == 0) {
    s.rank_work = 0u;
    s.arr_overflow = 0u;
  }

  // Rows of this CTA: t = blockIdx.x + k * gridDim.x.  Walking the 1024-row
  // chunks in order and taking the rows congruent to blockIdx.x in each
  // visits exactly this sequence, so the walk is chunk by chunk.
  const int G = (int)gridDim.x;
  int t = (int)blockIdx.x;
  if (t < T) src.issue(t, rowbuf);
  cp_async_commit();
  if (t + G < T) src.issue(t + G, rowbuf + words);
  cp_async_commit();

  for (int k = 0; t < T; ++k, t += G) {
    uint32_t* cur = rowbuf + (k & 1) * words;
    cp_async_wait<1>();
    __syncthreads();  // this row is staged; the previous row's state is reset

    // ---- L1: top-11-bit histogram; constant-bit masks per key class -----
    uint32_t keys[kFastItems], invs[kFastItems], slot[kFastItems];
    uint32_t lor[3] = {0u, 0u, 0u}, land[3] = {~0u, ~0u, ~0u};
    uint32_t ior[3] = {0u, 0u, 0u}, iand[3] = {~0u, ~0u, ~0u};
#pragma unroll
    for (int j = 0; j < kFastItems; ++j) {
      const int i = tid + j * kThreads;
      keys[j] = 0u;
      invs[j] = 0u;
      if (i < n) {
        const uint32_t kk = score_key(cur[i]);
        const uint32_t u = src.inv(cur, i);
        keys[j] = kk;
        invs[j] = u;
        atomicAdd(&s.table[kk >> 21], 1u);
        const uint32_t lo = kk & 0x1FFFFFu;
        const int c = key_class(kk);
#pragma unroll
        for (int e = 0; e < 3; ++e) {
          if (c == e) {
            lor[e] |= lo;
            land[e] &= lo;
            ior[e] |= u;
            iand[e] &= u;
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      lor[e] = __reduce_or_sync(0xFFFFFFFFu, lor[e]);
      land[e] = __reduce_and_sync(0xFFFFFFFFu, land[e]);
      ior[e] = __reduce_or_sync(0xFFFFFFFFu, ior[e]);
      iand[e] = __reduce_and_sync(0xFFFFFFFFu, iand[e]);
    }
    if (lane < 3) {
      // lane e publishes class e (all lanes hold the reduced values)
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        if (lane == e) {
          atomicOr(&s.acc_or[e], lor[e]);
          atomicAnd(&s.acc_and[e], land[e]);
          atomicOr(&s.acc_or[3 + e], ior[e]);
          atomicAnd(&s.acc_and[3 + e], iand[e]);
        }
      }
    }
    __syncthreads();

    // ---- SCAN1: bins in descending order; (buckets << 16 | count) packed --
    {
      const int bA = kHistBins - 1 - 2 * tid;
      const int bB = bA - 1;
      const uint32_t hA = s.table[bA], hB = s.table[bB];
      const uint32_t fA = fine_buckets(hA), fB = fine_buckets(hB);
      const uint32_t v = ((fA + fB) << 16) | (hA + hB);
      const uint32_t incl = warp_inclusive_scan(v);
      if (lane == 31) s.wa[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const uint32_t w = s.wa[lane];
        s.wb[lane] = warp_inclusive_scan(w) - w;
      }
      __syncthreads();
      const uint32_t ex = s.wb[warp] + incl - v;
      const uint32_t cA = ex & 0xFFFFu, gA = ex >> 16;
      const uint32_t cB = cA + hA, gB = gA + fA;
      const uint32_t need = (uint32_t)ksel;
      if (hA != 0u && cA < need && need <= cA + hA) {
        s.b1 = (uint32_t)bA;
        s.nfine = gA + fA;
      } else if (hB != 0u && cB < need && need <= cB + hB) {
        s.b1 = (uint32_t)bB;
        s.nfine = gB + fB;
      }
      if (hA != 0u) s.table[bA] = (gA << 8) | (uint32_t)(31 - __clz(fA));
      if (hB != 0u) s.table[bB] = (gB << 8) | (uint32_t)(31 - __clz(fB));
    }
    __syncthreads();

    // ---- L2: fine buckets for bins >= b1 ---------------------------------
    {
      const uint32_t b1 = s.b1;
      // Within key class c, the low 21 key bits below tz[c] are the same for
      // every candidate, and so are the bits of ~id at or above ib[c]; the
      // remaining bits, key bits first, order the candidates of one bin.
      int tz[3], ib[3];
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        const uint32_t vk = s.acc_or[e] ^ s.acc_and[e];
        const uint32_t vi = s.acc_or[3 + e] ^ s.acc_and[3 + e];
        tz[e] = vk ? min(__ffs(vk) - 1, 21) : 21;
        ib[e] = vi ? 32 - __clz(vi) : 0;
      }
#pragma unroll
      for (int j = 0; j < kFastItems; ++j) {
        const int i = tid + j * kThreads;
        slot[j] = kNoBucket;
        if (i < n && (keys[j] >> 21) >= b1) {
          const uint32_t tb = s.table[keys[j] >> 21];
          const int q = (int)(tb & 0xFFu);
          const int c = key_class(keys[j]);
          const int tzc = c == 0 ? tz[0] : (c == 1 ? tz[1] : tz[2]);
          const int ibc = c == 0 ? ib[0] : (c == 1 ? ib[1] : ib[2]);
          const uint32_t imask = ibc >= 32 ? 0xFFFFFFFFu : ((1u << ibc) - 1u);
          const int w = (21 - tzc) + ibc;
          const unsigned long long r =
              ((unsigned long long)((keys[j] & 0x1FFFFFu) >> tzc) << ibc) | (invs[j] & imask);
          const uint32_t sub = w >= q ? (uint32_t)(r >> (w - q)) : (uint32_t)(r << (q - w));
          const uint32_t g = (tb >> 8) + ((1u << q) - 1u - sub);
          atomicAdd(&s.fcnt[g], w <= q ? 0x10001u : 1u);
          slot[j] = g;
        }
      }
    }
    __syncthreads();

    // ---- SCAN2: bucket starts; can this row be ranked in place? ----------
    {
      const uint32_t nf = s.nfine;
      uint32_t c[3], ex3[3];
      uint32_t sum = 0u;
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        const uint32_t g = (uint32_t)(3 * tid + e);
        const uint32_t raw = g < nf ? s.fcnt[g] : 0u;
        c[e] = raw & 0xFFFFu;
        ex3[e] = raw >> 16;
        sum += c[e];
      }
      const uint32_t incl = warp_inclusive_scan(sum);
      if (lane == 31) s.wa[warp] = incl;
      __syncthreads();
      if (warp == 0) {
        const uint32_t w = s.wa[lane];
        s.wb[lane] = warp_inclusive_scan(w) - w;
      }
      __syncthreads();
      uint32_t st = s.wb[warp] + incl - sum;
      uint32_t work = 0u, over = 0u;
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        const uint32_t g = (uint32_t)(3 * tid + e);
        if (g < nf) {
          const bool exact = ex3[e] != 0u;
          s.fst[g] = st | (c[e] << 15) | (exact ? 0x80000000u : 0u);
          s.fcnt[g] = 0u;
          if (st < (uint32_t)ksel && !exact && c[e] > 1u) {
            work += c[e] * c[e];
            if (st + c[e] > (uint32_t)(ksel + kArrSlack)) over = 1u;
          }
          st += c[e];
        }
      }
      work = __reduce_add_sync(0xFFFFFFFFu, work);
      over = __reduce_or_sync(0xFFFFFFFFu, over);
      if (lane == 0 && (work | over)) {
        atomicAdd(&s.rank_work, work);
        atomicOr(&s.arr_overflow, over);
      }
      // L1/L2 state is no longer read in this row: reset it for the next.
      for (int i = tid; i < kHistBins; i += kThreads) s.table[i] = 0u;
      if (tid < 6) {
        s.acc_or[tid] = 0u;
        s.acc_and[tid] = 0xFFFFFFFFu;
      }
    }
    __syncthreads();

    float* os = out_scores + (size_t)t * (size_t)K;
    int32_t* oi = out_ids + (size_t)t * (size_t)K;
    const bool fast = s.arr_overflow == 0u && s.rank_work <= kRankLimit;

    if (fast) {
      // ---- SCATTER: bucket members that can still be winners, into arr --
      const uint32_t kcap = (uint32_t)(ksel + kArrSlack);
#pragma unroll
      for (int j = 0; j < kFastItems; ++j) {
        if (slot[j] != kNoBucket) {
          const uint32_t g = slot[j];
          const uint32_t meta = s.fst[g];
          const uint32_t st = meta & 0x7FFFu;
          const bool exact = (meta >> 31) != 0u;
          uint32_t pos = kNoBucket;
          if (st < (uint32_t)ksel) {
            pos = st + atomicAdd(&s.fcnt[g], 1u);
            if (pos < (exact ? (uint32_t)ksel : kcap))
              s.arr[pos] = ((unsigned long long)keys[j] << 32) | invs[j];
            else
              pos = kNoBucket;
          }
          slot[j] = pos == kNoBucket ? kNoBucket : (g | (pos << 16));
        }
      }
      __syncthreads();
      // The staged row is consumed: stream the row after next into it.
      if (t + 2 * G < T) src.issue(t + 2 * G, cur);
      cp_async_commit();
      for (int i = tid; i < kFineMax; i += kThreads) s.fcnt[i] = 0u;
      if (tid == 0) {
        s.rank_work = 0u;
        s.arr_overflow = 0u;
      }

      // ---- RANK: position = bucket start + members with a larger key -----
#pragma unroll
      for (int j = 0; j < kFastItems; ++j) {
        if (slot[j] != kNoBucket) {
          const uint32_t g = slot[j] & 0xFFFFu;
          const uint32_t pos = slot[j] >> 16;
          const uint32_t meta = s.fst[g];
          const uint32_t st = meta & 0x7FFFu;
          const uint32_t cnt = (meta >> 15) & 0x7FFFu;
          uint32_t fin = pos;
          if ((meta >> 31) == 0u && cnt > 1u) {
            const unsigned long long mine = ((unsigned long long)keys[j] << 32) | invs[j];
            uint32_t r = 0u;
            for (uint32_t e = st; e < st + cnt; ++e) {
              const unsigned long long o = s.arr[e];
              r += (o > mine || (o == mine && e < pos)) ? 1u : 0u;
            }
            fin = st + r;
          }
          if (fin < (uint32_t)ksel) {
            s.out_s[fin] = score_bits(keys[j]);
            s.out_i[fin] = src.out_id(t, invs[j]);
          }
        }
      }
      __syncthreads();

      // ---- STORE ----------------------------------------------------------
      for (int j = tid; j < K; j += kThreads) {
        if (j < ksel) {
          os[j] = __uint_as_float(s.out_s[j]);
          oi[j] = s.out_i[j];
        } else {
          os[j] = __uint_as_float(0xFF800000u);
          oi[j] = -1;
        }
      }
    } else {
      // ---- Fallback: radix select + sort on the staged row ---------------
      int n_pow2 = 1;
      while (n_pow2 < ksel) n_pow2 <<= 1;
      select_sort_row(
          s.sel, n, ksel, s.arr, n_pow2, [&](int i) { return score_key(cur[i]); },
          [&](int i) { return src.inv(cur, i); });
      for (int j = tid; j < K; j += kThreads) {
        if (j < ksel) {
          const unsigned long long w = s.arr[j];
          os[j] = __uint_as_float(score_bits((uint32_t)(w >> 32)));
          oi[j] = src.out_id(t, (uint32_t)w);
        } else {
          os[j] = __uint_as_float(0xFF800000u);
          oi[j] = -1;
        }
      }
      __syncthreads();  // every read of the staged row, arr and `fast` is done
      if (t + 2 * G < T) src.issue(t + 2 * G, cur);
      cp_async_commit();
      if (tid == 0) {
        s.rank_work = 0u;
        s.arr_overflow = 0u;
      }
    }
  }
  cp_async_wait<0>();
}

inline size_t fast_smem_bytes(int staged_words) {
  const size_t words = (size_t)((staged_words + 3) & ~3);
  return ((sizeof(FastShared) + 15) & ~(size_t)15) + 2 * words * sizeof(uint32_t);
}

}  // namespace dcp
