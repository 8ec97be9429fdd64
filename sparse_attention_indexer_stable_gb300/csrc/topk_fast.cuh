// topk_fast.cuh -- the streaming top-K path for rows of up to 16384
// candidates and K <= 4096 (the merge at DCP=4, K=2048, the local top-K over
// 4096 columns and the fused top-K over all shards fall here).
//
// A persistent grid walks the rows: CTAs of 512 threads, two per SM, for many
// rows (while one CTA waits at a barrier or on a copy the other computes), or
// 1024-thread CTAs, one per row or per SM, for few, long or large-K rows.  A
// row's scores and ids are staged in shared memory by bulk copies (TMA) read
// straight from the rank-major layout, on separate barriers; the next row's
// scores are copied as soon as L1 has read this row's.  Selection and final
// order come out of one two-level bucket pass instead of a radix select
// followed by a sort:
//
//  L1       a histogram of the score keys' top 12 bits (11 in 1024-thread
//           CTAs) over every candidate: the "radix pass over 32-bit score
//           keys first" of "[Kernel] Optimize CuTeDSL DCP top-k merge",
//           Summary.
//  SCAN1    locates the bin b1 holding the K-th largest key (bins above it
//           are all winners) and gives every bin >= b1 a number of fine
//           buckets, about one per two keys, and a first bucket.
//  COMPACT  the candidates of bins >= b1 ("live", about K of them) are packed
//           into a dense list of 64-bit keys score_key<<32 | ~id.
//  L2       each live key's fine bucket: its bin's first bucket plus the top
//           bits of its key below the bin, skipping bits equal for all live
//           keys; the token id enters only where scores tie, which is the
//           page's conditional tie-break.  Buckets are numbered in key order.
//  SCAN2    a prefix sum over bucket sizes gives each bucket its first output
//           position.
//  SCATTER  keys of buckets that start before K go to their bucket's slice of
//           the list.
//  RANK     per list position: output position = bucket start + the bucket's
//           members with larger keys; positions >= K are the losers.  Buckets
//           hold a few keys, so this one step both finishes the selection at
//           the threshold and sorts the winners.  A warp's positions are
//           consecutive, so its output stores are nearly coalesced.
//
// Rows whose live set or buckets come out too large for this (pathologically
// clustered keys) take the radix-select + sort of topk_core.cuh on the same
// row (read again from global memory): the result never depends on the
// data's distribution, only the speed does.  Rows whose K-th key is -inf
// land there too and take a shorter way (fallback_row): merge rows with fewer
// real candidates than K, the rest padding (-inf, -1) from shards shorter than
// K, and masked rows of logits with fewer finite values than K.
//
// Barriers: shared state is reset only after the barrier that follows its last
// reader in the row (the race the first page's review reports came from
// resetting shared state that late warps had not yet read).
#pragma once

#include <cstddef>
#include <cstdint>

#include "topk_core.cuh"

namespace dcp {

constexpr int kStreamMaxN = 8192;             // candidates per row (two CTAs per SM)
constexpr int kStreamMaxNWide = 16384;        // candidates per row (one CTA per SM)
constexpr int kStreamMaxK = 2048;             // K of the regular instantiations
constexpr int kStreamMaxKWide = 4096;         // K of the one-CTA-per-row instantiation for larger K
constexpr uint32_t kNegInfKey = 0x007FFFFFu;  // score key of -inf: padding's, with ~id 0
constexpr uint32_t kBigBucket = 255;          // a larger bucket starting before K sends the row to the fallback
constexpr uint32_t kNone = 0xFFFFFFFFu;
constexpr unsigned long long kStageWaitLimit = 1ull << 31;  // cycles (about 1 s) to wait for a row's copy
constexpr uint32_t kStatusCopyTimeout = 1u;     // device status bit: a staging copy timed out
constexpr uint32_t kStatusBadShardAlignment = 2u;  // device status bit: a shard not 16-byte aligned

// Per-row sizes for a CTA of NT threads selecting up to KMAX winners.
// - The 512-thread CTAs walk many rows two to an SM: their L1 bins are the
//   score keys' top 12 bits, which keeps the live set near K even for
//   bf16-valued scores, and their shared memory is tighter: a live list of
//   2560 keys (a fuller threshold bin is refined first) and 2560 fine buckets
//   (at most 512 per L1 bin).
// - The 1024-thread CTAs (one row each, or rows of up to 16384 candidates)
//   use 11-bit bins, KMAX + 1024 live keys and as many fine buckets (at most
//   1024 per bin): a smaller histogram to scan and reset per row.
// Capacities are multiples of NT.
template <int NT, int KMAX = kStreamMaxK>
struct StreamCaps {
  static constexpr int kL1Bits = NT == 512 ? 12 : 11;
  static constexpr int kL1Shift = 32 - kL1Bits;
  static constexpr int kL1Bins = 1 << kL1Bits;
  static constexpr uint32_t kLowMask = (1u << kL1Shift) - 1u;  // key bits below the L1 bin
  static constexpr int kRefShift = kL1Shift - 11;  // the refinement digit: 11 bits below the bin
  static constexpr uint32_t kPadBin = kNegInfKey >> kL1Shift;  // bin of -inf keys (padding)
  static constexpr int kLive = NT == 512 ? 2560 : KMAX + 1024;
  static constexpr int kFine = NT == 512 ? 2560 : KMAX + 1024;
  // fine buckets per L1 bin; the bins above b1 hold fewer than K keys and
  // get fewer than K buckets, so a row needs fewer than kFine
  static constexpr uint32_t kBinBuckets = (uint32_t)(kFine - KMAX);
  // list positions: up to the end of the bucket straddling K
  static constexpr int kRankMax = KMAX + 256;
  // RANK's scratch in the aux region: rank keys (u64) then bucket info (u16)
  // per list position
  static constexpr int kScratchWords = (kRankMax * 8 + kRankMax * 2 + 15) / 16 * 4;
};

template <int LIVE, int FINE, int BINS>
struct StreamShared {
  unsigned long long live[LIVE];      // live keys; then in bucket order; fallback: sorted winners
  uint32_t fine[FINE];                // L2 sizes, then start << 16 | size << 8 | fill cursor
  union {
    uint32_t table[BINS];             // L1 counts, then first bucket << 8 | log2(buckets)
    SelectShared sel;                 // the fallback's radix-select state
  } u;
  uint32_t wa[kMaxWarps];
  uint32_t wb[kMaxWarps];
  // per warp (plain stores, reduced where they are read: no same-address
  // atomics from every warp)
  uint32_t wraw[kMaxWarps];           // OR of the raw scores' bits below the bin
  uint32_t wior[kMaxWarps];           // OR of ~ids (not 0)
  uint32_t wiand[kMaxWarps];          // AND of ~ids (not 0)
  uint32_t live_cursor;
  uint32_t b1;                        // L1 bin of the K-th largest key
  uint32_t above_b1;                  // candidates in bins above b1
  uint32_t found_digit, found_above, found_count;  // refinement of b1
  uint32_t p_end;                     // end of the bucket straddling the slice's end
  uint32_t p_begin;                   // start of the bucket straddling the slice's start
  uint32_t part_bh, part_bl;          // the slice's highest and lowest L1 bins
  uint32_t part_pmin, part_fmin;      // the first position and fine bucket of bin part_bh
  uint32_t part_pend, part_fend;      // the end position and fine bucket of bin part_bl
  uint32_t overflow;                  // a bucket to rank is too large
  uint32_t pad_n;                     // fallback: padding keys of the row
  uint32_t lscal[8];                  // list_sort's scalars
  unsigned long long stage_bar;       // completes when a row's scores land in the stage
  unsigned long long ids_bar;         // completes when a row's ids land in the aux region
};
template <int NT, int KMAX = kStreamMaxK>
using StreamSharedFor = StreamShared<StreamCaps<NT, KMAX>::kLive, StreamCaps<NT, KMAX>::kFine,
                                     StreamCaps<NT, KMAX>::kL1Bins>;

// 16-byte vector accesses to these arrays need 16-byte aligned offsets.
template <class S, int FINE>
constexpr bool stream_layout_ok() {
  return offsetof(S, live) % 16 == 0 && offsetof(S, fine) % 16 == 0 &&
         offsetof(S, u) == offsetof(S, fine) + sizeof(uint32_t) * FINE &&  // one region to reset
         offsetof(S, stage_bar) % 8 == 0;
}
template <int NT, int KMAX>
constexpr bool stream_caps_ok() {
  using C = StreamCaps<NT, KMAX>;
  return stream_layout_ok<StreamSharedFor<NT, KMAX>, C::kFine>() && C::kLive % NT == 0 &&
         C::kFine % NT == 0 && C::kFine >= 2048 /* the refinement histogram */ &&
         C::kLive >= KMAX && C::kRankMax >= KMAX + (int)kBigBucket - 1;
}
static_assert(stream_caps_ok<512, kStreamMaxK>(), "caps");
static_assert(stream_caps_ok<1024, kStreamMaxK>(), "caps");
static_assert(stream_caps_ok<1024, kStreamMaxKWide>(), "caps");

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// mbarrier and 1-D bulk-copy (TMA) primitives.  One thread arms the barrier
// with the byte count of a row and issues the row's copies; every thread then
// waits on the barrier's phase.
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global to shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_1d(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Marks the rows t, t + G, ... < T of a CTA that stops after a copy timed
// out: every slot gets id DCP_ID_UNWRITTEN and a NaN score, so that a
// caller who does not check the device status cannot mistake stale memory
// for a result.  Every thread of the CTA calls it.
__device__ __forceinline__ void mark_rows_unwritten(float* out_scores, int32_t* out_ids, int t, int T,
                                                 int G, int K) {
  for (; t < T; t += G) {
    float* os = out_scores + (size_t)t * (size_t)K;
    int32_t* oi = out_ids + (size_t)t * (size_t)K;
    for (int j = threadIdx.x; j < K; j += blockDim.x) {
      os[j] = __uint_as_float(0x7FFFFFFFu);  // NaN
      oi[j] = INT32_MIN;                      // DCP_ID_UNWRITTEN
    }
  }
}

// Waits for phase `parity` of `bar` to complete, giving up once `limit`
// SM clock cycles have passed (each poll returns within a bounded time, so
// the wait is bounded).  Returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  unsigned long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = clock64();
  while (clock64() - t0 < limit)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Programmatic dependent launch: wait until the stream's previous grid has
// completed and its memory is visible (a no-op when the launch did not allow
// overlap), then let the next grid be scheduled.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Fine buckets for an L1 bin of h candidates: half of h rounded up to a power
// of two, at least 1 and at most cap (a power of two; 0 for an empty bin).
// Never more than h, so the bins above b1 (fewer than K candidates) get fewer
// than K buckets.
__device__ __forceinline__ uint32_t fine_buckets(uint32_t h, uint32_t cap) {
  const uint32_t p = (1u << (32 - __clz(h - 1u))) >> 1;  // next power of two >= h, halved
  return h == 0u ? 0u : min(max(p, 1u), cap);
}

// Loads P consecutive histogram words at p (ascending bins) into h in
// descending bin order.
template <int P>
__device__ __forceinline__ void load_bins_desc(const uint32_t* p, uint32_t (&h)[P]) {
  if constexpr (P % 4 == 0 && P > 4) {
#pragma unroll
    for (int g = 0; g < P / 4; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(p + 4 * g);
      h[P - 1 - 4 * g] = w.x;
      h[P - 2 - 4 * g] = w.y;
      h[P - 3 - 4 * g] = w.z;
      h[P - 4 - 4 * g] = w.w;
    }
  } else if constexpr (P == 4) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    h[0] = w.w;
    h[1] = w.z;
    h[2] = w.y;
    h[3] = w.x;
  } else if constexpr (P == 2) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    h[0] = w.y;
    h[1] = w.x;
  } else {
#pragma unroll
    for (int e = 0; e < P; ++e) h[e] = p[P - 1 - e];
  }
}

// Digit d of a 2048-bin histogram with above(d) < need <= above(d) + hist[d]
// (above(d): total of the bins above d).  wa/wb: per-warp scratch.  One
// thread writes the results; the caller synchronises before reading them.
template <int NT>
__device__ __forceinline__ void find_digit_desc(const uint32_t* hist, uint32_t need, uint32_t* wa,
                                                uint32_t* wb, uint32_t& digit, uint32_t& above_out,
                                                uint32_t& count_out) {
  constexpr int kPer = kHistBins / NT;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t h[kPer];
  load_bins_desc<kPer>(hist + kHistBins - kPer * (tid + 1), h);
  uint32_t local = 0u;
#pragma unroll
  for (int e = 0; e < kPer; ++e) local += h[e];
  const uint32_t incl = warp_inclusive_scan(local);
  if (lane == 31) wa[warp] = incl;
  row_sync();
  if (warp == 0) {
    const uint32_t w = lane < NT / 32 ? wa[lane] : 0u;
    wb[lane] = warp_inclusive_scan(w) - w;
  }
  row_sync();
  uint32_t above = wb[warp] + incl - local;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    if (h[e] != 0u && above < need && need <= above + h[e]) {
      digit = (uint32_t)(kHistBins - 1 - (kPer * tid + e));
      above_out = above;
      count_out = h[e];
    }
    above += h[e];
  }
}

// Shared-memory bytes of the streaming kernel with NT threads: the state, the
// stage for a row's `score_words` scores, and the aux region (the row's
// `ids_words` ids when they are staged, RANK's scratch after COMPACT; the
// larger of the two).  The stage and the aux region start on 128-byte
// boundaries: bulk copies into a destination that was only 16-byte aligned
// measured slower (decode merge 5.66 -> 5.60 us per launch, 5.41 -> 5.21 us
// per graph replay; fused top-K of one row 6.58 -> 6.34 us).
template <int NT, int KMAX = kStreamMaxK>
inline size_t stream_smem_bytes(int score_words, int ids_words) {
  constexpr int kScratch = StreamCaps<NT, KMAX>::kScratchWords;
  const int aux = ids_words > kScratch ? ids_words : kScratch;
  return ((sizeof(StreamSharedFor<NT, KMAX>) + 127) & ~(size_t)127) +
         (size_t)((score_words + 31) & ~31) * 4 + (size_t)((aux + 3) & ~3) * 4;
}

// Orders this thread's earlier shared-memory writes before later bulk copies
// (async proxy) into the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Zeroes `words` (a multiple of 4) 16-byte-aligned shared words.
template <int NT>
__device__ __forceinline__ void zero_words(uint32_t* p, int words) {
  for (int i = 4 * (int)threadIdx.x; i < words; i += 4 * NT)
    *reinterpret_cast<uint4*>(p + i) = make_uint4(0u, 0u, 0u, 0u);
}

// Scratch of list_sort: pointers into the calling kernel's shared memory.
struct ListScratch {
  const unsigned long long* list;  // the keys score_key << 32 | ~id (read only)
  uint32_t* fine;                  // >= the list's length (bucket sizes)
  uint32_t* table;                 // the histogram: 2^kBits words
  unsigned long long* rk;          // >= w + 255 keys (the bucket-ordered list)
  uint16_t* info;                  // as many entries: bucket size << 8 | slot
  uint32_t* wa;                    // 32 words
  uint32_t* wb;                    // 32 words
  uint32_t* scal;                  // 8 words
};

// Sorts the top w of the m keys list[0, m) (no padding among them;
// 0 < w <= m <= kCap) and hands them, in order, to out(position, key):
// the bucket machinery of the row kernels applied to a list.  A histogram of
// the keys' top kBits bits locates the bin of the w-th key; the bins at or
// above it get buckets in position space (bin b owns buckets
// [above(b), above(b) + count(b))), each key going to the bucket named by the
// top bits of y = (key bits below the bin >> tzf) << ibf | (~id low ibf bits),
// tzf and ibf taken from the list itself, so a list of -inf keys, whose
// score bits are all equal, is ordered by its ids alone; a bucket's members
// are ranked by comparing their keys, identical keys (outside the contract)
// by their slots.  Every thread of the CTA calls it; returns false, having
// output nothing, if a bucket to rank holds more than 255 keys (keys that
// agree on every bit the buckets use).
template <int NT, int kBits, int kCap, class Out>
__device__ bool list_sort(const ListScratch& ls, int m, int w, Out out) {
  constexpr int kWarpsT = NT / 32;
  constexpr int kShift = 32 - kBits;
  constexpr uint32_t kLowMask = (1u << kShift) - 1u;
  constexpr int kBins = 1 << kBits;
  constexpr int kWindows = kBins / 128;
  constexpr int kPer = (kCap + NT - 1) / NT;
  static_assert(kWindows <= 32, "one lane per window");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* table = ls.table;
  uint32_t* fine = ls.fine;
  uint32_t& b1_s = ls.scal[0];
  uint32_t& nsel_s = ls.scal[1];
  uint32_t& p_end_s = ls.scal[2];
  uint32_t& over_s = ls.scal[3];
  uint32_t& ro_s = ls.scal[4];
  uint32_t& ior_s = ls.scal[5];
  uint32_t& iand_s = ls.scal[6];
  if (w <= 0 || m < w || m > kCap) return w <= 0;  // uniform

  zero_words<NT>(fine, (m + 3) & ~3);
  zero_words<NT>(table, kBins);
  if (tid == 0) {
    p_end_s = over_s = ro_s = ior_s = 0u;
    iand_s = 0xFFFFFFFFu;
  }
  row_sync();
  {
    uint32_t raw_or = 0u, ior = 0u, iand = 0xFFFFFFFFu;
    for (int e = tid; e < m; e += NT) {
      const unsigned long long lk = ls.list[e];
      const uint32_t kk = (uint32_t)(lk >> 32);
      atomicAdd(&table[kk >> kShift], 1u);
      raw_or |= score_bits(kk);
      ior |= (uint32_t)lk;
      iand &= (uint32_t)lk;
    }
    raw_or = __reduce_or_sync(0xFFFFFFFFu, raw_or & kLowMask);
    ior = __reduce_or_sync(0xFFFFFFFFu, ior);
    iand = __reduce_and_sync(0xFFFFFFFFu, iand);
    if (lane == 0) {
      atomicOr(&ro_s, raw_or);
      atomicOr(&ior_s, ior);
      atomicAnd(&iand_s, iand);
    }
  }
  row_sync();
  // bin totals per window of 128 bins
  for (int win = warp; win < kWindows; win += kWarpsT) {
    const uint4 h4 = *reinterpret_cast<const uint4*>(table + 128 * win + 4 * lane);
    const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, h4.x + h4.y + h4.z + h4.w);
    if (lane == 0) ls.wb[win] = sum;
  }
  row_sync();
  // every warp scans the window totals (high to low) and ranks the bins of
  // its windows at or above the w-th key: above | count << 13 | q << 26
  {
    const uint32_t wt = lane < kWindows ? ls.wb[kWindows - 1 - lane] : 0u;
    const uint32_t wincl = warp_inclusive_scan(wt);
    for (int win = warp; win < kWindows; win += kWarpsT) {
      const uint32_t above_w = __shfl_sync(0xFFFFFFFFu, wincl - wt, kWindows - 1 - win);
      const uint32_t tot_w = __shfl_sync(0xFFFFFFFFu, wt, kWindows - 1 - win);
      if (tot_w == 0u || above_w >= (uint32_t)w) continue;
      const int hi = 128 * win + 127;
      uint32_t h[4];
      load_bins_desc<4>(table + (hi - 4 * lane - 3), h);
      const uint32_t local = h[0] + h[1] + h[2] + h[3];
      const uint32_t incl = warp_inclusive_scan(local);
      uint32_t a = above_w + incl - local;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (h[e] != 0u && a < (uint32_t)w) {
          const int b = hi - 4 * lane - e;
          if ((uint32_t)w <= a + h[e]) {
            b1_s = (uint32_t)b;
            nsel_s = a + h[e];
          }
          const uint32_t q = h[e] > 1u ? 32u - __clz(h[e] - 1u) : 0u;
          table[b] = a | (h[e] << 13) | (q << 26);
        }
        a += h[e];
      }
    }
  }
  row_sync();
  const uint32_t b1 = b1_s;
  const uint32_t nsel = nsel_s;  // keys in bins >= b1: they take the buckets
  const uint32_t ro = ro_s;
  const uint32_t vi = ior_s ^ iand_s;
  const int tzf = ro ? min(__ffs(ro) - 1, kShift) : kShift;
  const int ibf = vi ? 32 - __clz(vi) : 0;
  const uint32_t imask = ibf >= 32 ? 0xFFFFFFFFu : ((1u << ibf) - 1u);
  const int wf = kShift - tzf + ibf;
  uint32_t gsl[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * NT;
    gsl[u] = kNone;
    if (e < m) {
      const unsigned long long lk = ls.list[e];
      const uint32_t kk = (uint32_t)(lk >> 32);
      if ((kk >> kShift) >= b1) {
        const uint32_t tb = table[kk >> kShift];
        const int q = (int)(tb >> 26);
        const unsigned long long y =
            ((unsigned long long)((kk & kLowMask) >> tzf) << ibf) | ((uint32_t)lk & imask);
        const uint32_t sub = wf >= q ? (uint32_t)(y >> (wf - q)) : (uint32_t)(y << (q - wf));
        const uint32_t cb = (tb >> 13) & 0x1FFFu;
        const uint32_t g = dbg_clamp((tb & 0x1FFFu) + cb - 1u - ((sub * cb) >> q), nsel);
        atomicAdd(&fine[g], 1u);
        gsl[u] = g;
      }
    }
  }
  row_sync();
  // bucket starts over [0, nsel)
  {
    uint32_t local = 0u;
    uint32_t c[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int g = kPer * tid + u;
      c[u] = g < (int)nsel ? fine[g] : 0u;
      local += c[u];
    }
    const uint32_t incl = warp_inclusive_scan(local);
    if (lane == 31) ls.wa[warp] = incl;
    row_sync();
    const uint32_t wt = lane < kWarpsT ? ls.wa[lane] : 0u;
    const uint32_t wti = warp_inclusive_scan(wt);
    uint32_t st = __shfl_sync(0xFFFFFFFFu, wti - wt, warp) + incl - local;
    uint32_t over = 0u;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int g = kPer * tid + u;
      if (g < (int)nsel) {
        fine[g] = (st << 16) | (min(c[u], 255u) << 8);
        if (st < (uint32_t)w) {
          if (c[u] > kBigBucket) over = 1u;
          if ((uint32_t)w <= st + c[u]) p_end_s = st + c[u];
        }
      }
      st += c[u];
    }
    over = __reduce_or_sync(0xFFFFFFFFu, over);
    if (lane == 0 && over) over_s = 1u;
  }
  row_sync();
  if (over_s != 0u) return false;
  // the keys of buckets starting before w into their bucket's slots
  const uint32_t p_cap = (uint32_t)w + kBigBucket;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (gsl[u] != kNone) {
      const uint32_t old = atomicAdd(&fine[gsl[u]], 1u);
      if ((old >> 16) < (uint32_t)w) {
        const uint32_t pos = dbg_clamp((old >> 16) + (old & 0xFFu), p_cap);
        ls.info[pos] = (uint16_t)(old & 0xFFFFu);
        ls.rk[pos] = ls.list[tid + u * NT];
      }
    }
  }
  row_sync();
  // rank within the bucket: the members with larger keys, and identical
  // keys in earlier slots
  const uint32_t p_end = min(p_end_s, p_cap);
  for (uint32_t p = tid; p < p_end; p += NT) {
    const uint32_t inf = ls.info[p];
    const uint32_t slot = inf & 0xFFu;
    const uint32_t st = dbg_clamp(p - slot, p + 1u);
    const uint32_t cnt = dbg_clamp(inf >> 8, p_cap + 1u - st);
    const unsigned long long mine = ls.rk[p];
    uint32_t r = 0u;
    for (uint32_t e = 0; e < cnt; ++e) {
      const unsigned long long x = ls.rk[st + e];
      r += (x > mine || (x == mine && e < slot)) ? 1u : 0u;
    }
    const uint32_t fin = st + r;
    if (fin < (uint32_t)w) out(fin, mine);
  }
  row_sync();
  return true;
}

// The fallback for one row of the streaming kernel: the row again from
// global memory, radix select + sort (topk_core.cuh).  Two kinds of rows
// whose K-th key is -inf take a shorter way:
// - merge rows with fewer candidates above the padding key than K, the rest
//   padding (-inf, -1) from shards shorter than K (alike keys, so too large a
//   bucket for the fast path): just those candidates are sorted and the tail
//   padded;
// - rows of logits with fewer finite values than K (a masked row), where ids
//   grow with the candidate index: the finite candidates are sorted, and the
//   -inf winners, the lowest ids among the -inf candidates, are the first
//   ones in index order, so a running count places them.
// Out of line: rare, and its code stays out of the row loop.  Every thread of
// the CTA calls it; the staged ids are intact (only SCATTER overwrites them).
template <int NT, int KMAX, class Source, class Shared>
__device__ __noinline__ void fallback_row(const Source src, Shared& s, const uint32_t* aux, int t,
                                          int n, int ksel, int K, float* os, int32_t* oi) {
  using Caps = StreamCaps<NT, KMAX>;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n4 = n >> 2;
  int nwin = ksel;  // winners in s.live[0, nwin), sorted
  int tail = ksel;  // padding from here on (positions nwin .. tail are written)
  bool sorted = false;
  // list_sort's scratch: the table and bucket arrays, RANK's scratch in the
  // aux region (the staged ids are read before it is written)
  unsigned long long* lrk = reinterpret_cast<unsigned long long*>(const_cast<uint32_t*>(aux));
  const ListScratch ls{s.live, s.fine, s.u.table, lrk,
                       reinterpret_cast<uint16_t*>(lrk + Caps::kRankMax), s.wa, s.wb, s.lscal};
  const uint32_t rbase0 = src.row_base(t);
  auto out_at = [&](uint32_t pos, unsigned long long key) {
    os[pos] = __uint_as_float(score_bits((uint32_t)(key >> 32)));
    oi[pos] = src.out_id_from(rbase0, (uint32_t)key);
  };
  if constexpr (Source::kStagesIds) {
    if (s.b1 == Caps::kPadBin) {
      if (tid == 0) s.live_cursor = 0u;  // COMPACT's last use was barriers ago
      row_sync();
      uint32_t npad = 0u;
#pragma unroll 1
      for (int c0 = 0; c0 < n4; c0 += NT) {
        const int c = c0 + tid;
        uint4 k4 = make_uint4(0u, 0u, 0u, 0u), u4 = k4;
        if (c < n4) {
          k4 = src.key4_global(t, c);
          u4 = src.inv4(aux, c);
        }
        const uint32_t ks[4] = {k4.x, k4.y, k4.z, k4.w};
        const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
        uint32_t m = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (c < n4) {
            if (ks[e] > kNegInfKey || (ks[e] == kNegInfKey && us[e] != 0u)) m |= 1u << e;
            npad += (ks[e] == kNegInfKey && us[e] == 0u) ? 1u : 0u;
          }
        }
        const uint32_t cnt = __popc(m);
        const uint32_t incl = warp_inclusive_scan(cnt);
        uint32_t base = 0u;
        if (lane == 31) base = atomicAdd(&s.live_cursor, incl);
        uint32_t slot = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (m & (1u << e)) {
            if (slot < (uint32_t)Caps::kLive) s.live[slot] = ((unsigned long long)ks[e] << 32) | us[e];
            ++slot;
          }
        }
      }
      npad = __reduce_add_sync(0xFFFFFFFFu, npad);
      if (lane == 0 && npad != 0u) atomicAdd(&s.pad_n, npad);
      row_sync();
      const uint32_t nreal = s.live_cursor;  // candidates above the padding key
      if (nreal < (uint32_t)ksel && nreal + s.pad_n >= (uint32_t)ksel &&
          list_sort<NT, Caps::kL1Bits, Caps::kLive>(ls, (int)nreal, (int)nreal, out_at)) {
        nwin = 0;  // the winners are written; padding from nreal on
        tail = (int)nreal;
        sorted = true;
      }
    }
  } else {
    if (s.b1 == Caps::kPadBin && src.index_ordered()) {
      if (tid == 0) {
        s.live_cursor = 0u;
        s.pad_n = 0u;  // here: the -inf candidates
      }
      row_sync();
      uint32_t ninf = 0u;
#pragma unroll 1
      for (int c0 = 0; c0 < n4; c0 += NT) {
        const int c = c0 + tid;
        uint32_t ks[4] = {0u, 0u, 0u, 0u};
        if (c < n4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) ks[e] = src.key_global(t, 4 * c + e);
        }
        const uint4 u4 = src.inv4(aux, c);
        const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
        uint32_t m = 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (c < n4) {
            if (ks[e] > kNegInfKey) m |= 1u << e;
            ninf += ks[e] == kNegInfKey ? 1u : 0u;
          }
        }
        const uint32_t cnt = __popc(m);
        const uint32_t incl = warp_inclusive_scan(cnt);
        uint32_t base = 0u;
        if (lane == 31) base = atomicAdd(&s.live_cursor, incl);
        uint32_t slot = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (m & (1u << e)) {
            if (slot < (uint32_t)Caps::kLive) s.live[slot] = ((unsigned long long)ks[e] << 32) | us[e];
            ++slot;
          }
        }
      }
      ninf = __reduce_add_sync(0xFFFFFFFFu, ninf);
      if (lane == 0 && ninf != 0u) atomicAdd(&s.pad_n, ninf);
      row_sync();
      const uint32_t nf = s.live_cursor;  // candidates above -inf
      if (nf < (uint32_t)ksel && nf + s.pad_n >= (uint32_t)ksel) {
        // the first ksel - nf -inf candidates in index order take positions
        // nf .. ksel
        constexpr int kWarpsT = NT / 32;
        const int warp = tid >> 5;
        const uint32_t need = (uint32_t)ksel - nf;
        const uint32_t rbase = src.row_base(t);
        uint32_t before = 0u;  // -inf candidates in earlier chunks
#pragma unroll 1
        for (int c0 = 0; c0 < n4 && before < need; c0 += NT) {
          const int c = c0 + tid;
          uint32_t f = 0u;
          if (c < n4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) f |= (src.key_global(t, 4 * c + e) == kNegInfKey ? 1u : 0u) << e;
          }
          const uint32_t cnt = __popc(f);
          const uint32_t incl = warp_inclusive_scan(cnt);
          if (lane == 31) s.wa[warp] = incl;
          row_sync();
          const uint32_t wt = lane < kWarpsT ? s.wa[lane] : 0u;
          const uint32_t wti = warp_inclusive_scan(wt);
          const uint32_t chunk = __shfl_sync(0xFFFFFFFFu, wti, kWarpsT - 1);
          uint32_t q = before + __shfl_sync(0xFFFFFFFFu, wti - wt, warp) + incl - cnt;
          if (f != 0u) {
            const uint4 u4 = src.inv4(aux, c);
            const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (f & (1u << e)) {
                if (q < need) {
                  os[nf + q] = __uint_as_float(0xFF800000u);  // -inf
                  oi[nf + q] = src.out_id_from(rbase, us[e]);
                }
                ++q;
              }
            }
          }
          before += chunk;
          row_sync();  // s.wa is rewritten by the next chunk
        }
        if (list_sort<NT, Caps::kL1Bits, Caps::kLive>(ls, (int)nf, (int)nf, out_at)) {
          nwin = 0;  // the finite winners are written, the -inf ones above
          tail = ksel;
          sorted = true;
        }
      }
    }
  }
  if (!sorted) {
    int n_pow2 = 1;
    while (n_pow2 < ksel) n_pow2 <<= 1;
    select_sort_row<NT>(
        s.u.sel, n, ksel, s.live, n_pow2, [&](int i) { return src.key_global(t, i); },
        [&](int i) { return src.inv_global(t, i); });
  }
  const uint32_t rbase = src.row_base(t);
  for (int j = tid; j < K; j += NT) {
    if (j < nwin) {
      const unsigned long long w = s.live[j];
      os[j] = __uint_as_float(score_bits((uint32_t)(w >> 32)));
      oi[j] = src.out_id_from(rbase, (uint32_t)w);
    } else if (j >= tail) {
      os[j] = __uint_as_float(0xFF800000u);  // -inf
      oi[j] = -1;
    }
  }
}

// kSplit: the grid's y dimension splits each row's sort into gridDim.y
// parts.  Part y (a CTA of its own) stages the whole row and selects its
// threshold bin (the same in every part), then sorts only the bins whose
// output positions meet its slice [y*slice, (y+1)*slice) of the
// k = min(K, n) winners (the last part's slice ending at k) and writes that
// slice.  The slices partition the output, so a row's result does not
// depend on the split.
template <int NT, int MAXN, int KMAX, class Source, bool kSplit>
__global__ void __launch_bounds__(NT, NT == 1024 ? 1 : 2)
    topk_stream_kernel(Source src, int T, int K, int slice, float* __restrict__ out_scores,
                       int32_t* __restrict__ out_ids, unsigned int* __restrict__ status) {
  constexpr int kWarpsT = NT / 32;
  constexpr int kVec = MAXN / 4 / NT;  // 16-byte score chunks per thread
  constexpr int kItems = 4 * kVec;
  using Caps = StreamCaps<NT, KMAX>;
  using Shared = StreamSharedFor<NT, KMAX>;
  constexpr int kRankMax = Caps::kRankMax;
  constexpr int kLiveMax = Caps::kLive;
  constexpr int kFineMax = Caps::kFine;
  constexpr int kL1Bins = Caps::kL1Bins;
  constexpr int kL1Shift = Caps::kL1Shift;
  constexpr uint32_t kLowMask = Caps::kLowMask;
  constexpr int kRefShift = Caps::kRefShift;
  constexpr uint32_t kPadBin = Caps::kPadBin;
  constexpr int kLivePer = kLiveMax / NT;
  constexpr int kFinePer = kFineMax / NT;
  constexpr int kBinsPer = kL1Bins / NT;

  extern __shared__ __align__(16) unsigned char smem_raw[];
  Shared& s = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* stage =
      reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(Shared) + 127) & ~(size_t)127));
  const int n = src.count();  // multiple of 4, <= MAXN
  uint32_t* aux = stage + ((n + 31) & ~31);  // the row's ids (when staged), then RANK's scratch
  unsigned long long* rkl = reinterpret_cast<unsigned long long*>(aux);
  uint16_t* info = reinterpret_cast<uint16_t*>(rkl + kRankMax);
  const int n4 = n >> 2;
  const int ksel = K < n ? K : n;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  // Shared-memory set-up first: it touches no global memory, so it may run
  // while the stream's previous kernel is still finishing.
  zero_words<NT>(s.fine, kFineMax + kL1Bins);  // fine and the table behind it
  if (tid == 0) {
    s.live_cursor = 0u;
    s.p_end = s.p_begin = 0u;
    s.overflow = 0u;
    s.pad_n = 0u;
  }

  // This CTA's rows are t = blockIdx.x + k * gridDim.x: walking the rows in
  // chunks of 1024 and taking, in each, the rows congruent to blockIdx.x
  // visits exactly this sequence.
  const int G = (int)gridDim.x;
  int t = (int)blockIdx.x;
  // this part's output slice [lo, hi)
  const uint32_t lo = kSplit ? blockIdx.y * (uint32_t)slice : 0u;
  const uint32_t hi =
      kSplit && blockIdx.y + 1u < gridDim.y ? lo + (uint32_t)slice : (uint32_t)ksel;
  if (tid == 0) {
    mbar_init(&s.stage_bar, 1u);
    mbar_init(&s.ids_bar, 1u);
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();  // every thread, before its first global access
  if constexpr (Source::kIndirect) {
    // separate shards: their 16-byte alignment is only visible here
    if (!__syncthreads_and(tid != 0 || src.shards_aligned())) {
      if (tid == 0) atomicOr(status, kStatusBadShardAlignment);
      mark_rows_unwritten(out_scores, out_ids, t, T, G, K);
      return;
    }
  }
  if (tid == 0) {
    if (t < T) {
      src.issue_scores(t, stage, &s.stage_bar);
      if constexpr (Source::kStagesIds) src.issue_ids(t, aux, &s.ids_bar);
    }
  }

  for (uint32_t k = 0; t < T; t += G, ++k) {
    const bool staged = mbar_wait_bounded(&s.stage_bar, k & 1u, kStageWaitLimit);
    // the row is staged (or its copy timed out) and the previous row's state reset
    if (__syncthreads_or(!staged)) {
      // Report the timeout, mark this CTA's rows unwritten and stop; first
      // give the copies a last, bounded chance to land.  If one never lands
      // the CTA still exits (nothing waits forever); such a copy could only
      // write into this CTA's shared memory.
      if (tid == 0) atomicOr(status, kStatusCopyTimeout);
      mbar_wait_bounded(&s.stage_bar, k & 1u, kStageWaitLimit);
      if constexpr (Source::kStagesIds) mbar_wait_bounded(&s.ids_bar, k & 1u, kStageWaitLimit);
      mark_rows_unwritten(out_scores, out_ids, t, T, G, K);
      return;
    }
    dbg_skew();
    // The copy of the next row's scores into the stage starts as soon as this
    // row's are consumed (after L1); its ids follow at the end of the row (the
    // aux region serves RANK until then) and are needed only by COMPACT.

    // ---- L1: histogram of the score keys' top bits -------------------------
    // Also ORs the raw scores' bits below the bin: the bits that are zero in
    // all of them are constant in every key of one sign (bf16-valued scores
    // leave the low 16 zero), which the buckets below skip.
    uint32_t keys[kItems];
    uint32_t raw_or = 0u;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const int c = tid + v * NT;
      if (c < n4) {
        const uint4 w = *reinterpret_cast<const uint4*>(stage + 4 * c);
        raw_or |= w.x | w.y | w.z | w.w;
        keys[4 * v + 0] = score_key(w.x);
        keys[4 * v + 1] = score_key(w.y);
        keys[4 * v + 2] = score_key(w.z);
        keys[4 * v + 3] = score_key(w.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) atomicAdd(&s.u.table[keys[4 * v + e] >> kL1Shift], 1u);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) keys[4 * v + e] = 0u;
      }
    }
    raw_or = __reduce_or_sync(0xFFFFFFFFu, raw_or & kLowMask);
    if (lane == 0) s.wraw[warp] = raw_or;
    row_sync();
    // L1 was the last reader of the staged scores (the rest of the row works
    // from the keys in registers, the staged ids and, in the fallback, global
    // memory): stream the next row's scores in behind the rest of this one.
    const bool next_issued = t + G < T;
    if (tid == 0 && next_issued) src.issue_scores(t + G, stage, &s.stage_bar);

    // ---- SCAN1: bins high to low; packed (buckets << 16 | candidates) -------
    // A warp whose bins are all empty (most warps: the keys fill a narrow
    // band of bins) only reports a zero total.
    {
      uint32_t h[kBinsPer], f[kBinsPer];
      load_bins_desc<kBinsPer>(s.u.table + kL1Bins - kBinsPer * (tid + 1), h);
      uint32_t any = 0u;
#pragma unroll
      for (int e = 0; e < kBinsPer; ++e) any |= h[e];
      const bool warp_busy = __any_sync(0xFFFFFFFFu, any != 0u);
      uint32_t local = 0u, incl = 0u;
      if (warp_busy) {
#pragma unroll
        for (int e = 0; e < kBinsPer; ++e) {
          f[e] = fine_buckets(h[e], Caps::kBinBuckets);
          local += (f[e] << 16) | h[e];
        }
        incl = warp_inclusive_scan(local);
      }
      if (lane == 31) s.wa[warp] = incl;
      row_sync();
      if (warp_busy) {
        // every warp scans the per-warp totals itself (no second barrier)
        const uint32_t wt = lane < kWarpsT ? s.wa[lane] : 0u;
        const uint32_t wti = warp_inclusive_scan(wt);
        uint32_t ex = __shfl_sync(0xFFFFFFFFu, wti - wt, warp) + incl - local;
#pragma unroll
        for (int e = 0; e < kBinsPer; ++e) {
          const uint32_t above = ex & 0xFFFFu, fabove = ex >> 16;
          // this and the thread's later bins lie below b1: no table entries
          if (above >= (uint32_t)ksel) break;
          const int b = kL1Bins - 1 - (kBinsPer * tid + e);
          if (h[e] != 0u) {
            if (above < (uint32_t)ksel && (uint32_t)ksel <= above + h[e]) {
              s.b1 = (uint32_t)b;
              s.above_b1 = above;
            }
            // the bins holding the slice's first and last positions
            if (kSplit && above <= lo && lo < above + h[e]) {
              s.part_bh = (uint32_t)b;
              s.part_pmin = above;
              s.part_fmin = fabove;
            }
            if (above < hi && hi <= above + h[e]) {
              s.part_bl = (uint32_t)b;
              s.part_pend = above + h[e];
              s.part_fend = fabove + f[e];
            }
            s.u.table[b] = (fabove << 8) | (uint32_t)(31 - __clz(f[e]));
          }
          ex += (f[e] << 16) | h[e];
        }
      }
    }
    if constexpr (Source::kStagesIds) {
      // COMPACT reads the row's ids: they were copied during L1 and SCAN1
      const bool ids_ok = mbar_wait_bounded(&s.ids_bar, k & 1u, kStageWaitLimit);
      if (__syncthreads_or(!ids_ok)) {
        // also let the next row's scores, already on their way, land
        if (tid == 0) atomicOr(status, kStatusCopyTimeout);
        mbar_wait_bounded(&s.ids_bar, k & 1u, kStageWaitLimit);
        if (next_issued) mbar_wait_bounded(&s.stage_bar, (k + 1u) & 1u, kStageWaitLimit);
        mark_rows_unwritten(out_scores, out_ids, t, T, G, K);
        return;
      }
      dbg_skew();
    } else {
      row_sync();
    }

    const uint32_t b1 = s.b1;
    // The slice's bins are [bl, bh] (all bins >= b1 without a split); their
    // positions start at pmin and their fine buckets at fmin, which the
    // slice's lists and buckets count from.
    const uint32_t bh = kSplit ? s.part_bh : 0u, bl = s.part_bl;
    const uint32_t pmin = kSplit ? s.part_pmin : 0u, fmin = kSplit ? s.part_fmin : 0u;
    const int nfine = (int)(s.part_fend - fmin);
    uint32_t nlv = s.part_pend - pmin;  // the slice's live candidates
    // Live candidates are those with bin <= bh and (key >> kRefShift) >=
    // live_from.  Normally that is every candidate of bins [bl, bh]; when the
    // live set would overflow the live list and bl is b1, the next 11 key
    // bits of bin b1 are histogrammed (in `fine`, still zero) and only its
    // candidates from the digit holding the K-th key on are kept live.
    uint32_t live_from = bl << 11;
    if (nlv > (uint32_t)kLiveMax && bl == b1) {
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        if ((tid + (j >> 2) * NT) < n4 && (keys[j] >> kL1Shift) == b1)
          atomicAdd(&s.fine[(keys[j] >> kRefShift) & 0x7FFu], 1u);
      }
      row_sync();
      find_digit_desc<NT>(s.fine, (uint32_t)ksel - s.above_b1, s.wa, s.wb, s.found_digit,
                          s.found_above, s.found_count);
      row_sync();
      live_from |= s.found_digit;
      nlv = s.above_b1 + s.found_above + s.found_count - pmin;
      if constexpr (kPoisonBuild) {
        row_sync();
        dbg_poison<NT>(s.fine, kHistBins);
        __syncthreads();
      }
      zero_words<NT>(s.fine, kHistBins);  // the refinement histogram: 2048 words of fine
      row_sync();
    }
    const int nlive = (int)nlv;
    bool fast = nlive <= kLiveMax;

    // ---- COMPACT: live candidates into a dense list -------------------------
    if (fast) {
      uint32_t mask = 0u;
      const uint32_t lf = live_from << kRefShift;  // live: key >= lf (and bin <= bh)
      // kSplit: key - lf < span <=> lf <= key < (bh + 1) << kL1Shift (mod 2^32)
      const uint32_t span = ((bh + 1u) << kL1Shift) - lf;
      if (lf != 0u) {
        // candidates past the row hold key 0 (< lf)
        if constexpr (kSplit) {
#pragma unroll
          for (int j = 0; j < kItems; ++j) mask |= (keys[j] - lf < span ? 1u : 0u) << j;
        } else {
#pragma unroll
          for (int j = 0; j < kItems; ++j) mask |= (keys[j] >= lf ? 1u : 0u) << j;
        }
      } else {
#pragma unroll
        for (int j = 0; j < kItems; ++j)
          mask |= ((tid + (j >> 2) * NT) < n4 && (!kSplit || (keys[j] >> kL1Shift) <= bh) ? 1u : 0u)
                  << j;
      }
      const uint32_t cnt = __popc(mask);
      const uint32_t incl = warp_inclusive_scan(cnt);
      uint32_t base = 0u;
      if (lane == 31 && incl != 0u) base = atomicAdd(&s.live_cursor, incl);  // warps with live keys
      unsigned long long* dst =
          s.live + dbg_clamp(__shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt, kLiveMax + 1u - cnt);
      if constexpr (Source::kStagesIds) {
        // OR / AND of the inverted ids around the live candidates (padding's
        // ~id of 0 left out: it is the smallest, so ordering on the varying
        // bits alone still puts it last)
        uint32_t ior = 0u, iand = 0xFFFFFFFFu;
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
          if ((tid + v * NT) < n4) {
            const uint4 u4 = src.inv4(aux, tid + v * NT);
            const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ior |= us[e];
              iand &= us[e] ? us[e] : 0xFFFFFFFFu;
              if (mask & (1u << (4 * v + e)))
                *dst++ = ((unsigned long long)keys[4 * v + e] << 32) | us[e];
            }
          }
        }
        ior = __reduce_or_sync(0xFFFFFFFFu, ior);
        iand = __reduce_and_sync(0xFFFFFFFFu, iand);
        if (lane == 0) {
          s.wior[warp] = ior;
          s.wiand[warp] = iand;
        }
      } else {
        // ids computed from the candidate index (below n): only the live
        // candidates' are formed; their statistics are known (L2)
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
          if (((mask >> (4 * v)) & 0xFu) != 0u) {
            const uint4 u4 = src.inv4(aux, tid + v * NT);
            const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (mask & (1u << (4 * v + e)))
                *dst++ = ((unsigned long long)keys[4 * v + e] << 32) | us[e];
          }
        }
      }
    }
    row_sync();

    // ---- L2: fine bucket of every live candidate ---------------------------
    unsigned long long lkey[kLivePer];
    uint32_t gslot[kLivePer];
    if (fast) {
      // For finite scores the key bits below the L1 bin and below tzf are
      // equal within a sign, and the bits of ~id at or above ibf are equal for
      // every live candidate (but padding), so within one bin keys are
      // ordered like y = (low key bits >> tzf) << ibf | (~id low ibf bits), a
      // wf-bit number whose top q bits name the bucket.  Bins up to kPadBin
      // (-inf, where padding lives, and below) keep every bit.
      const uint32_t ro = __reduce_or_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wraw[lane] : 0u);
      // ~id bits that vary: measured in COMPACT, or, for ids computed from
      // the candidate index i < n, the low bits of n - 1 (~i agrees above them)
      const uint32_t vi = Source::kStagesIds
                              ? __reduce_or_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wior[lane] : 0u) ^
                                    __reduce_and_sync(0xFFFFFFFFu,
                                                      lane < kWarpsT ? s.wiand[lane] : 0xFFFFFFFFu)
                          : n > 1            ? 0xFFFFFFFFu >> __clz(n - 1)
                                             : 0u;
      const int tzf = ro ? min(__ffs(ro) - 1, kL1Shift) : kL1Shift;
      const int ibf = vi ? 32 - __clz(vi) : 0;
      const uint32_t imask = ibf >= 32 ? 0xFFFFFFFFu : ((1u << ibf) - 1u);
      const int wf = kL1Shift - tzf + ibf;
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        const int e = tid + u * NT;
        gslot[u] = kNone;
        lkey[u] = 0ull;
        if (e < nlive) {
          lkey[u] = s.live[e];
          const uint32_t k = (uint32_t)(lkey[u] >> 32);
          const uint32_t inv = (uint32_t)lkey[u];
          const uint32_t bin = k >> kL1Shift;
          const uint32_t tb = s.u.table[bin];
          const int q = (int)(tb & 0xFFu);
          unsigned long long y;
          int w;
          if (bin > kPadBin) {
            y = ((unsigned long long)((k & kLowMask) >> tzf) << ibf) | (inv & imask);
            w = wf;
          } else {
            y = ((unsigned long long)(k & kLowMask) << 32) | inv;
            w = kL1Shift + 32;
          }
          const uint32_t sub = w >= q ? (uint32_t)(y >> (w - q)) : (uint32_t)(y << (q - w));
          const uint32_t g = (tb >> 8) + ((1u << q) - 1u - sub) - fmin;
          atomicAdd(&s.fine[dbg_clamp(g, kFineMax)], 1u);
          gslot[u] = dbg_clamp(g, kFineMax);
        }
      }
    }
    row_sync();

    // ---- SCAN2: bucket starts ------------------------------------------------
    // fine[g] becomes start << 16 | min(size, 255) << 8, its low byte the
    // fill cursor for SCATTER.
    if (fast) {
      // warps whose buckets all lie past the last one only report a zero total
      const bool warp_busy = kFinePer * 32 * warp < nfine;
      // buckets past nfine are empty (fine is zero there), so no guards
      uint32_t c[kFinePer];
      uint32_t local = 0u, incl = 0u;
      uint32_t* my = s.fine + kFinePer * tid;
      if (warp_busy) {
        if constexpr (kFinePer % 2 == 0) {
#pragma unroll
          for (int e = 0; e < kFinePer; e += 2) {
            const uint2 w = *reinterpret_cast<const uint2*>(my + e);
            c[e] = w.x;
            c[e + 1] = w.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kFinePer; ++e) c[e] = my[e];
        }
#pragma unroll
        for (int e = 0; e < kFinePer; ++e) local += c[e];
        incl = warp_inclusive_scan(local);
      }
      if (lane == 31) s.wa[warp] = incl;
      row_sync();
      if (warp_busy) {
        const uint32_t wt = lane < kWarpsT ? s.wa[lane] : 0u;
        const uint32_t wti = warp_inclusive_scan(wt);
        uint32_t st = __shfl_sync(0xFFFFFFFFu, wti - wt, warp) + incl - local;
        uint32_t over = 0u;
        uint32_t w[kFinePer];
        // the slice's positions, counted from pmin
        const uint32_t klo = lo - pmin, khi = hi - pmin;
#pragma unroll
        for (int e = 0; e < kFinePer; ++e) {
          w[e] = (st << 16) | (min(c[e], 255u) << 8);
          if (st < khi && (!kSplit || klo < st + c[e])) {
            if (c[e] > kBigBucket) over = 1u;
            if (khi <= st + c[e]) s.p_end = st + c[e];
            if (kSplit && st <= klo) s.p_begin = st;
          }
          st += c[e];
        }
        if constexpr (kFinePer % 2 == 0) {
#pragma unroll
          for (int e = 0; e < kFinePer; e += 2)
            *reinterpret_cast<uint2*>(my + e) = make_uint2(w[e], w[e + 1]);
        } else {
#pragma unroll
          for (int e = 0; e < kFinePer; ++e) my[e] = w[e];
        }
        over = __reduce_or_sync(0xFFFFFFFFu, over);
        if (lane == 0 && over) s.overflow = 1u;
      }
    }
    row_sync();
    fast = fast && s.overflow == 0u;

    float* os = out_scores + (size_t)t * (size_t)K;
    int32_t* oi = out_ids + (size_t)t * (size_t)K;
    if (fast) {
      // ---- SCATTER: winners' keys into the list, in bucket order -----------
      // Members of buckets that start before K go to their bucket's slots.
      // Per list position the aux region records the bucket's size << 8 | the
      // slot and, for shared buckets, rank_key(key, slot) =
      // key << 11 | (255 - slot): members of a bucket share their key's top
      // 11 or 12 bits (the L1 bin), so dropping 11 of them keeps the key order
      // within the bucket, identical keys told apart by their slot (the
      // smaller slot first).
      const uint32_t klo = lo - pmin, khi = hi - pmin;
      const uint32_t p_begin = kSplit ? s.p_begin : 0u;
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        if (gslot[u] != kNone) {
          const uint32_t old = atomicAdd(&s.fine[gslot[u]], 1u);
          // buckets meeting the slice, listed from the one holding its start
          if ((old >> 16) < khi && (!kSplit || klo < (old >> 16) + ((old >> 8) & 0xFFu))) {
            const uint32_t pos = dbg_clamp((old >> 16) - p_begin + (old & 0xFFu), kRankMax);
            s.live[pos] = lkey[u];
            info[pos] = (uint16_t)(old & 0xFFFFu);
            if (((old >> 8) & 0xFFu) > 1u) rkl[pos] = (lkey[u] << 11) | (255u - (old & 0xFFu));
          }
        }
      }
      row_sync();

      // ---- RANK: position = bucket start + members ranking above ----------
      // Per list position.  Consecutive positions share buckets, so a warp's
      // buckets are usually all small enough for a 4-wide window.
      const uint32_t p_end = min(s.p_end - p_begin, (uint32_t)kRankMax);
      const uint32_t rbase = src.row_base(t);
      const uint32_t p_off = pmin + p_begin;  // output position of list position 0
      for (uint32_t p = tid; p < p_end; p += NT) {
        const uint32_t inf = info[p];
        const uint32_t st = dbg_clamp(p - (inf & 0xFFu), p + 1u);
        const uint32_t cnt = dbg_clamp(inf >> 8, kRankMax + 8u - st);
        const unsigned long long key = s.live[p];
        const uint32_t mc = __reduce_max_sync(__activemask(), cnt);
        uint32_t r = 0u;
        if (mc > 1u) {
          const unsigned long long* b = rkl + st;
          const unsigned long long mine = rkl[p];
          if (mc <= 4u) {
#pragma unroll
            for (uint32_t e = 0; e < 4u; ++e)
              if (e < cnt && cnt > 1u) r += b[e] > mine ? 1u : 0u;
          } else if (mc <= 8u) {
#pragma unroll
            for (uint32_t e = 0; e < 8u; ++e)
              if (e < cnt && cnt > 1u) r += b[e] > mine ? 1u : 0u;
          } else if (cnt > 1u) {
            for (uint32_t e = 0; e < cnt; ++e) r += b[e] > mine ? 1u : 0u;
          }
        }
        const uint32_t fin = p_off + st + r;
        if ((!kSplit || lo <= fin) && fin < hi) {
          os[fin] = __uint_as_float(score_bits((uint32_t)(key >> 32)));
          oi[fin] = src.out_id_from(rbase, (uint32_t)key);
        }
      }
      if (!kSplit || blockIdx.y + 1u == gridDim.y) {
        for (int j = ksel + tid; j < K; j += NT) {
          os[j] = __uint_as_float(0xFF800000u);  // -inf
          oi[j] = -1;
        }
      }
    } else {
      fallback_row<NT, KMAX>(src, s, aux, t, n, ksel, K, os, oi);
    }
    // SCATTER wrote the aux region through ordinary stores; the next row's
    // ids are copied into it after the barrier.
    if constexpr (Source::kStagesIds) fence_proxy_async_shared();
    row_sync();  // every reader of this row's shared state is done
    if constexpr (Source::kStagesIds)
      if (tid == 0 && t + G < T) src.issue_ids(t + G, aux, &s.ids_bar);

    if constexpr (kPoisonBuild) {
      dbg_poison<NT>(s.fine, kFineMax + kL1Bins);
      dbg_poison<NT>(s.live, 2 * kLiveMax);
      dbg_poison<NT>(s.wa, 2 * kMaxWarps);
      dbg_poison<NT>(s.wraw, 3 * kMaxWarps);
      if constexpr (!Source::kStagesIds) dbg_poison<NT>(aux, Caps::kScratchWords);
      if (tid == 0) {
        s.b1 = s.above_b1 = 0xA5A5A5A5u;
        s.part_bh = s.part_bl = s.part_pmin = s.part_fmin = 0xA5A5A5A5u;
        s.part_pend = s.part_fend = 0xA5A5A5A5u;
        s.found_digit = s.found_above = s.found_count = 0xA5A5A5A5u;
      }
      __syncthreads();
    }
    zero_words<NT>(s.fine, kFineMax + kL1Bins);  // fine and the table behind it
    if (tid == 0) {
      s.live_cursor = 0u;
      s.p_end = s.p_begin = 0u;
      s.overflow = 0u;
      s.pad_n = 0u;
    }
  }
}

}  // namespace dcp
