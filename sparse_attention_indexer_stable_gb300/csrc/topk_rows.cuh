// topk_rows.cuh -- the many-row merge at K = 2048 (prefill-scale merges: more
// than two rows per SM, dcp <= 4 shards of 2048 candidates each).
//
// Four 256-thread CTAs share an SM, each walking the rows
// t = blockIdx.x + k*gridDim.x (the 1024-row chunks of "Reserve the sparse
// indexer's DCP top-k merge scratch through the workspace manager", Purpose,
// visited in order; rows are independent).  Four rows in flight per SM keep
// the SM busy while any one CTA sits in a short serial step of its row.  No
// row is staged in shared memory: each thread reads its 32 candidates with
// 16-byte coalesced loads straight from the rank-major (dcp, T, K) buffers,
// and the next row is prefetched into L2 about a third of a row ahead (early
// enough to land, late enough to stay: a whole row ahead it was evicted again
// and DRAM read 45% more than the candidates).  The 32 score keys of a thread
// wait in tensor memory from L1 to COMPACT, so the registers that held them
// take the row's ids, loaded during SCAN1.
//
// Per row ("[Kernel] Optimize CuTeDSL DCP top-k merge", Summary: a radix pass
// over 32-bit score keys first, the id tie-break only where scores tie):
//  L1       histogram of the score keys' top 12 bits (4096 bins).
//  SCAN1    every warp sums four 128-bin windows; every warp then scans the
//           32 window totals and ranks the bins of its windows at or above
//           the window holding the K-th key: bin b gets above(b), the number
//           of candidates in higher bins, and count(b).  The bin b1 with
//           above(b1) < K <= above(b1) + count(b1) holds the K-th key.
//  COMPACT  candidates of bins >= b1 ("live", about K + a part of b1) are
//           packed as 64-bit entries score_key << 32 | id (the id inverted
//           where it is used); the ids were loaded during SCAN1.  A bin b1
//           too full for the list is refined first on its next 11 key bits.
//  L2       buckets in position space: bin b owns buckets
//           [above(b), above(b) + count(b)), one per candidate, and each live
//           key goes to the bucket named by the top bits of its key below the
//           bin, the varying low bits of ~id joining only below equal score
//           bits (the conditional tie-break).  Buckets are numbered in key
//           order.
//  SCAN2    prefix sum of bucket sizes: each bucket's first output position.
//  SCATTER  keys of buckets starting before K take a slot in their bucket's
//           range, with a rank key that orders the bucket's members.
//  RANK     per list position: output position = bucket start + the members
//           ranking above; positions >= K are the losers.  A warp's positions
//           are consecutive, so its output stores are nearly coalesced.
//
// Rows whose buckets come out too large (more than 255 keys in one, e.g.
// keys clustered within a few ulps) or whose K-th key is in the -inf bin take
// the radix select + sort of topk_core.cuh on the same row (rows_fallback):
// the result never depends on the data's distribution, only the speed does.
//
// Barriers: shared state is reset only after the barrier that follows its
// last reader in the row (the race the first page's review reports came from
// resetting shared state that late warps had not yet read).
#pragma once

#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "topk_core.cuh"
#include "topk_fast.cuh"

namespace dcp {

constexpr int kRowsNT = 256;             // threads per CTA (four CTAs per SM)
constexpr int kRowsK = 2048;             // K of this kernel
constexpr int kRowsMaxN = 8192;          // candidates per row: dcp <= 4
constexpr int kRowsL1Shift = 20;         // L1 bins: the score key's top 12 bits
constexpr int kRowsBins = 4096;
constexpr int kRowsLive = 2560;          // live list (a fuller bin b1 is refined first)
constexpr int kRowsFine = kRowsLive;     // position-space buckets: one per live key
constexpr int kRowsRankMax = kRowsK + 256;  // list positions: up to the end of the bucket straddling K
constexpr int kRowsRankWords = (kRowsRankMax + 8) * 2;  // 64-bit rank keys, + a window's overrun
constexpr int kRowsRegionWords = kRowsRankWords + kRowsRankMax / 2;  // + u16 bucket info
constexpr uint32_t kRowsPadBin = kNegInfKey >> kRowsL1Shift;  // bin of -inf keys (padding)
constexpr int kRowsInfIds = kRowsFine + kRowsRegionWords;     // fallback: ~ids of -inf candidates

struct RowsShared {
  uint32_t fine[kRowsFine];            // L2 bucket sizes, then start << 16 | size << 8 | fill cursor
  uint32_t region[kRowsRegionWords];   // L1 histogram, then the bin table; after L2 RANK's scratch;
                                       // the fallback's radix-select state
  unsigned long long live[kRowsLive];  // live keys; the fallback's sorted winners
  uint32_t wa[kMaxWarps];
  uint32_t wb[kMaxWarps];              // SCAN1: window totals
  uint32_t wraw[kRowsNT / 32];         // per warp: OR of the raw scores' bits below the bin
  uint32_t wior[kRowsNT / 32];         // per warp: OR of ~ids
  uint32_t wiand[kRowsNT / 32];        // per warp: AND of ~ids (padding's 0 left out)
  uint32_t live_cursor;
  uint32_t b1;                         // L1 bin of the K-th largest key
  uint32_t nlive;                      // candidates in bins >= b1 (after refinement: live)
  uint32_t above_b1;                   // candidates in bins above b1
  uint32_t found_digit, found_above, found_count;  // refinement of b1
  uint32_t p_end;                      // end of the bucket straddling K
  uint32_t overflow;                   // a bucket to rank is too large
  uint32_t pad_cnt;                    // candidates in the -inf bin
  uint32_t pad_n;                      // fallback: padding candidates
  uint32_t lscal[8];                   // list_sort's scalars
  uint32_t tmem_base;                  // this CTA's tensor-memory columns
};
static_assert(offsetof(RowsShared, region) == sizeof(uint32_t) * kRowsFine,
              "fine and the histogram are one region to reset");
static_assert(offsetof(RowsShared, region) % 16 == 0 && offsetof(RowsShared, live) % 16 == 0,
              "16-byte vector accesses");
static_assert(kRowsRegionWords >= kRowsBins, "histogram");
static_assert(sizeof(SelectShared) <= sizeof(uint32_t) * kRowsRegionWords, "fallback state");
static_assert(kRowsLive >= kRowsK && kRowsRankMax >= kRowsK + (int)kBigBucket - 1, "caps");
// the fallback's -inf ~ids (one per candidate) fill fine and region; its
// radix histogram (256 words) follows at most K - 1 finite keys in live
static_assert(kRowsInfIds >= kRowsMaxN && 2 * (kRowsK - 1) + 256 <= 2 * kRowsLive, "fallback");

// Starts pulling `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// Tensor memory (TMEM) holds each thread's 32 score keys from L1 to COMPACT,
// which frees the registers that hold them for the row's id loads (issued
// right after L1, in flight through SCAN1).  A CTA allocates 64 columns once:
// warp w owns columns 32*(w/4) .. +31 of lane quarter w%4 (a warp reaches
// only its own quarter of the 128 lanes), one column per key.  Four CTAs per
// SM take 256 of the 512 columns, so an allocation never waits on this
// kernel's own CTAs (tcgen05.alloc blocks in hardware until columns are free;
// a kernel of another stream holding TMEM on the SM can only delay it).
__device__ __forceinline__ void tmem_alloc64(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 64;\n"
               ::"r"(smem_u32(dst)) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc64(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 64;\n" ::"r"(taddr) : "memory");
}
// A CTA barrier that also orders tensor-memory operations around it.
__device__ __forceinline__ void tmem_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// r[0..32) into columns taddr .. taddr+31 of the thread's lane; returns once
// the store has completed (the registers are free again).
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;\n"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Columns taddr .. taddr+7 of the thread's lane into r, waited for.
__device__ __forceinline__ void tmem_load8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

// A 16-byte read-only load that does not allocate in L1: each candidate is
// read once, and L1 (what shared memory leaves of it) then keeps the spilled
// registers instead (prefill 209.9 -> 209.1 us).
__device__ __forceinline__ uint4 ldg4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// The fallback for one row, the row read again from global memory.
// - A row whose K-th key is -inf (fewer finite candidates than K: shards
//   shorter than K padded with (-inf, -1), or masked rows whose local top-K
//   holds real -inf candidates): the finite candidates are all winners and
//   are sorted as a list; the next winners are the real -inf candidates with
//   the lowest ids (a radix select on the id first when there are more of
//   them than the list holds), sorted as a list; padding fills the rest.
// - Otherwise (buckets too large, or negative NaNs among the winners): the
//   radix select + sort of topk_core.cuh over the whole row.
// Out of line: rare, and its code stays out of the row loop.  Every thread
// of the CTA calls it.
template <class Source>
__device__ __noinline__ void rows_fallback(const Source src, RowsShared& s, int t, int n,
                                           float* os, int32_t* oi) {
  constexpr int NT = kRowsNT;
  constexpr int kWarpsT = NT / 32;
  constexpr int ksel = kRowsK;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n4 = n >> 2;
  const uint32_t rbase = src.row_base(t);
  SelectShared& sel = *reinterpret_cast<SelectShared*>(s.region);
  // list_sort's scratch: the histogram, then RANK's scratch, in the region
  const ListScratch ls{s.live, s.fine, s.region,
                       reinterpret_cast<unsigned long long*>(s.region),
                       reinterpret_cast<uint16_t*>(s.region + kRowsRankWords), s.wa, s.wb,
                       s.lscal};
  int off = 0;
  auto out_at = [&](uint32_t pos, unsigned long long key) {
    os[off + (int)pos] = __uint_as_float(score_bits((uint32_t)(key >> 32)));
    oi[off + (int)pos] = src.out_id_from(rbase, (uint32_t)key);
  };
  if (s.b1 == kRowsPadBin) {
    // One pass over the row: the finite candidates into the list, the real
    // -inf candidates' ~ids into inf_ids (fine and region, one array of
    // kRowsInfIds words: room for every candidate), padding counted.
    uint32_t* inf_ids = s.fine;
    if (tid == 0) {
      s.live_cursor = 0u;
      s.pad_n = 0u;
      s.found_count = 0u;  // here: the real -inf candidates
    }
    row_sync();
    uint32_t npad = 0u;
    uint32_t ior = 0u, iand = 0xFFFFFFFFu;  // over the real -inf candidates' ~ids
#pragma unroll 1
    for (int c0 = 0; c0 < n4; c0 += NT) {
      const int c = c0 + tid;
      uint4 k4 = make_uint4(0u, 0u, 0u, 0u), u4 = k4;
      if (c < n4) {
        k4 = src.key4_global(t, c);
        const uint4 i4 = src.ids4_global(t, c);
        u4 = make_uint4(~i4.x, ~i4.y, ~i4.z, ~i4.w);
      }
      const uint32_t ks[4] = {k4.x, k4.y, k4.z, k4.w};
      const uint32_t us[4] = {u4.x, u4.y, u4.z, u4.w};
      uint32_t fm = 0u, im = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (c < n4) {
          fm |= (ks[e] > kNegInfKey ? 1u : 0u) << e;
          const bool real_inf = ks[e] == kNegInfKey && us[e] != 0u;
          im |= (real_inf ? 1u : 0u) << e;
          npad += (ks[e] == kNegInfKey && us[e] == 0u) ? 1u : 0u;
          if (real_inf) {
            ior |= us[e];
            iand &= us[e];
          }
        }
      }
      const uint32_t fcnt = __popc(fm);
      const uint32_t fincl = warp_inclusive_scan(fcnt);
      uint32_t fbase = 0u;
      if (lane == 31 && fincl) fbase = atomicAdd(&s.live_cursor, fincl);
      uint32_t fslot = __shfl_sync(0xFFFFFFFFu, fbase, 31) + fincl - fcnt;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (fm & (1u << e)) {
          if (fslot < (uint32_t)kRowsLive) s.live[fslot] = ((unsigned long long)ks[e] << 32) | us[e];
          ++fslot;
        }
      }
      if (__any_sync(0xFFFFFFFFu, im != 0u)) {  // padding-only chunks skip this
        const uint32_t icnt = __popc(im);
        const uint32_t iincl = warp_inclusive_scan(icnt);
        uint32_t ibase = 0u;
        if (lane == 31) ibase = atomicAdd(&s.found_count, iincl);
        uint32_t islot = __shfl_sync(0xFFFFFFFFu, ibase, 31) + iincl - icnt;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (im & (1u << e)) {
            if (islot < (uint32_t)kRowsInfIds) inf_ids[islot] = us[e];
            ++islot;
          }
        }
      }
    }
    npad = __reduce_add_sync(0xFFFFFFFFu, npad);
    ior = __reduce_or_sync(0xFFFFFFFFu, ior);
    iand = __reduce_and_sync(0xFFFFFFFFu, iand);
    if (lane == 0) {
      if (npad != 0u) atomicAdd(&s.pad_n, npad);
      s.wior[warp] = ior;  // the main path's slots, free here
      s.wiand[warp] = iand;
    }
    row_sync();
    const uint32_t nfin = s.live_cursor;                        // finite candidates
    const uint32_t rinf = min(s.found_count, (uint32_t)kRowsInfIds);  // real -inf candidates
    const uint32_t npd = s.pad_n;                               // padding
    if (nfin < (uint32_t)ksel && nfin + rinf + npd >= (uint32_t)ksel) {
      // The -inf winners: the w2 real -inf candidates with the lowest ids,
      // i.e. the largest ~ids.  With more of them than that, an 8-bit radix
      // select on ~id in shared memory finds the threshold thr (and how many
      // keys equal to it to take: identical ids, outside the contract).
      const uint32_t w2 = min(rinf, (uint32_t)ksel - nfin);
      uint32_t thr = 0u, take_eq = 0u;  // every ~id is > 0: all of them when rinf == w2
      if (w2 < rinf) {
        uint32_t* hist = reinterpret_cast<uint32_t*>(s.live + nfin);  // 256 words after the list
        // bits every real -inf ~id shares (ids from a narrow range share
        // their top bits): digits made only of them are not histogrammed
        const uint32_t all_and = __reduce_and_sync(
            0xFFFFFFFFu, lane < kWarpsT ? s.wiand[lane] : 0xFFFFFFFFu);
        const uint32_t varies =
            __reduce_or_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wior[lane] : 0u) ^ all_and;
        uint32_t prefix = 0u, pmask = 0u, need = w2;
#pragma unroll 1
        for (int shift = 24; shift >= 0; shift -= 8) {
          if (((varies >> shift) & 0xFFu) == 0u) {  // uniform: the digit every value has
            prefix |= all_and & (0xFFu << shift);
            pmask |= 0xFFu << shift;
            continue;
          }
          for (int i = tid; i < 256; i += NT) hist[i] = 0u;
          row_sync();
          for (uint32_t i = tid; i < rinf; i += NT) {
            const uint32_t v = inf_ids[i];
            if ((v & pmask) == prefix) atomicAdd(&hist[(v >> shift) & 0xFFu], 1u);
          }
          row_sync();
          if (warp == 0) {
            // lane l: digits 255 - 8l .. 248 - 8l, high to low
            uint32_t h[8], local = 0u;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              h[e] = hist[255 - 8 * lane - e];
              local += h[e];
            }
            uint32_t above = warp_inclusive_scan(local) - local;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (h[e] != 0u && above < need && need <= above + h[e]) {
                s.found_digit = (uint32_t)(255 - 8 * lane - e);
                s.found_above = above;
              }
              above += h[e];
            }
          }
          row_sync();
          prefix |= s.found_digit << shift;
          pmask |= 0xFFu << shift;
          need -= s.found_above;
          row_sync();  // the scalars and the histogram are rewritten by the next pass
        }
        thr = prefix;
        take_eq = need;  // keys equal to thr to take (1 unless ids repeat)
        if (tid == 0) s.lscal[7] = 0u;  // their claim counter (list_sort uses lscal[0..6])
        row_sync();
      }
      // the -inf winners behind the finite keys: live[nfin, nfin + w2)
      if (w2 > 0u) {
        if (tid == 0) s.live_cursor = nfin;
        row_sync();
      }
      for (uint32_t i0 = 0; w2 > 0u && i0 < rinf; i0 += NT) {
        const uint32_t i = i0 + tid;
        bool in = false;
        uint32_t v = 0u;
        if (i < rinf) {
          v = inf_ids[i];
          in = v > thr || (v == thr && atomicAdd(&s.lscal[7], 1u) < take_eq);
        }
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, in);
        uint32_t base = 0u;
        if (lane == 0 && b) base = atomicAdd(&s.live_cursor, (uint32_t)__popc(b));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        const uint32_t slot = base + __popc(b & ((1u << lane) - 1u));
        if (in && slot < (uint32_t)kRowsLive) s.live[slot] = ((unsigned long long)kNegInfKey << 32) | v;
      }
      if (w2 > 0u) row_sync();
      // the finite keys sorted to positions [0, nfin), the -inf winners to
      // [nfin, nfin + w2) (list_sort's scratch reuses fine and region)
      bool ok = list_sort<NT, 12, kRowsLive>(ls, (int)nfin, (int)nfin, out_at);
      if (ok && w2 > 0u) {
        ListScratch ls2 = ls;
        ls2.list = s.live + nfin;
        off = (int)nfin;
        ok = list_sort<NT, 12, kRowsLive>(ls2, (int)w2, (int)w2, out_at);
      }
      if (ok) {
        for (int j = (int)(nfin + w2) + tid; j < ksel; j += NT) {
          os[j] = __uint_as_float(0xFF800000u);  // -inf
          oi[j] = -1;
        }
        return;
      }
    }
  }
  select_sort_row<NT>(
      sel, n, ksel, s.live, ksel, [&](int i) { return src.key_global(t, i); },
      [&](int i) { return src.inv_global(t, i); });
  for (int j = tid; j < ksel; j += NT) {
    const unsigned long long w = s.live[j];
    os[j] = __uint_as_float(score_bits((uint32_t)(w >> 32)));
    oi[j] = src.out_id_from(rbase, (uint32_t)w);
  }
}

// One CTA of kRowsNT threads per row at a time; grid <= 4 * SMs.  Thread tid
// owns 16-byte chunk v of the row for v < 2*dcp: shard v/2, chunk
// tid + 256*(v%2) of the shard's 2048 candidates.
template <class Source>
__global__ void __launch_bounds__(kRowsNT, 4)
    merge_rows_kernel(Source src, int T, float* __restrict__ out_scores,
                      int32_t* __restrict__ out_ids, unsigned int* __restrict__ status) {
  constexpr int NT = kRowsNT;
  constexpr int kWarpsT = NT / 32;          // 8
  constexpr int kVec = kRowsMaxN / 4 / NT;  // 16-byte chunks per thread: 8
  constexpr int kItems = 4 * kVec;          // candidates per thread: 32
  constexpr int kLivePer = kRowsLive / NT;  // 10
  constexpr int kFinePer = kRowsFine / NT;  // 10
  constexpr int kWindows = kRowsBins / 128;  // 32 windows of 128 bins
  constexpr int K = kRowsK;
  constexpr int ksel = kRowsK;
  constexpr int kL1Shift = kRowsL1Shift;
  constexpr uint32_t kLowMask = (1u << kL1Shift) - 1u;  // key bits below the bin
  constexpr int kRefShift = kL1Shift - 11;  // the refinement digit: 11 bits below the bin

  extern __shared__ __align__(16) unsigned char smem_raw[];
  RowsShared& s = *reinterpret_cast<RowsShared*>(smem_raw);
  uint32_t* table = s.region;
  // RANK's scratch in the region (free after L2): wide rows 64-bit rank keys
  // (with the list index) and 16-bit bucket info; narrow rows 32-bit rank
  // keys and 32-bit bucket info that also holds the L1 bin, from which RANK
  // rebuilds a winner's key and ~id without going back to the list.
  unsigned long long* rk64 = reinterpret_cast<unsigned long long*>(s.region);
  uint32_t* rk32 = s.region;
  uint32_t* info32 = s.region + kRowsRankMax + 8;  // bin << 16 | size << 8 | slot
  uint16_t* info = reinterpret_cast<uint16_t*>(s.region + kRowsRankWords);
  static_assert(2 * (kRowsRankMax + 8) <= kRowsRegionWords, "narrow RANK scratch");
  const int n = src.count();  // dcp * 2048
  const int n4 = n >> 2;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const size_t shard_stride = (size_t)T * (size_t)K;  // elements between shards

  // Shared-memory set-up first: it touches no global memory, so it may run
  // while the stream's previous kernel is still finishing.
  zero_words<NT>(s.fine, kRowsFine + kRowsBins);  // fine and the histogram behind it
  if (tid == 0) {
    s.live_cursor = 0u;
    s.p_end = 0u;
    s.overflow = 0u;
  }
  const int G = (int)gridDim.x;
  int t = (int)blockIdx.x;
  grid_dependency_wait();  // every thread, before its first global access
  if constexpr (Source::kIndirect) {
    // separate shards: their 16-byte alignment is only visible here
    if (!__syncthreads_and(tid != 0 || src.shards_aligned())) {
      if (tid == 0) atomicOr(status, kStatusBadShardAlignment);
      mark_rows_unwritten(out_scores, out_ids, t, T, G, K);
      return;
    }
  }
  if (warp == 0) tmem_alloc64(&s.tmem_base);
  tmem_sync();
  const uint32_t tkeys =
      s.tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(32 * (warp >> 2));
  if (tid == 0 && t < T) src.prefetch_row(t);

  for (; t < T; t += G) {
    // this thread's 16-byte chunk v of row t: shard v/2, chunk tid + 256*(v%2)
    auto score_chunk = [&](int v) -> const float* {
      if constexpr (Source::kIndirect)
        return src.score_row(t, v >> 1) + 4 * (tid + NT * (v & 1));
      else
        return src.scores + (size_t)t * K + (size_t)(v >> 1) * shard_stride + 4 * (tid + NT * (v & 1));
    };
    auto id_chunk = [&](int v) -> const int32_t* {
      if constexpr (Source::kIndirect)
        return src.id_row(t, v >> 1) + 4 * (tid + NT * (v & 1));
      else
        return src.ids + (size_t)t * K + (size_t)(v >> 1) * shard_stride + 4 * (tid + NT * (v & 1));
    };
    uint4 w[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v)
      w[v] = (tid + v * NT) < n4 ? ldg4(score_chunk(v)) : make_uint4(0u, 0u, 0u, 0u);
    row_sync();  // the previous row's shared state is reset

    // ---- L1: histogram of the score keys' top 12 bits ----------------------
    // Also ORs the raw scores' bits below the bin: the bits that are zero in
    // all of them are constant in every key of one sign (bf16-valued scores
    // leave the low 16 zero), which the buckets below skip.
    uint32_t keys[kItems];
    uint32_t raw_or = 0u;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      if ((tid + v * NT) < n4) {  // uniform across the CTA: v < 2*dcp
        raw_or |= w[v].x | w[v].y | w[v].z | w[v].w;
        keys[4 * v + 0] = score_key(w[v].x);
        keys[4 * v + 1] = score_key(w[v].y);
        keys[4 * v + 2] = score_key(w[v].z);
        keys[4 * v + 3] = score_key(w[v].w);
#pragma unroll
        for (int e = 0; e < 4; ++e) atomicAdd(&table[keys[4 * v + e] >> kL1Shift], 1u);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) keys[4 * v + e] = 0u;
      }
    }
    raw_or = __reduce_or_sync(0xFFFFFFFFu, raw_or & kLowMask);
    if (lane == 0) s.wraw[warp] = raw_or;
    // the keys to tensor memory; the row's ids into the registers they held,
    // in flight through SCAN1 (predicated loads, none behind a branch)
    tmem_store32(tkeys, keys);
    uint4 ivs[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v)
      ivs[v] = (tid + v * NT) < n4 ? ldg4(id_chunk(v)) : make_uint4(0u, 0u, 0u, 0u);
    row_sync();

    // ---- SCAN1a: candidates per window of 128 bins (warp w: windows 4w..4w+3)
#pragma unroll
    for (int j = 0; j < kWindows / kWarpsT; ++j) {
      const int win = warp * (kWindows / kWarpsT) + j;
      const uint4 h4 = *reinterpret_cast<const uint4*>(table + 128 * win + 4 * lane);
      const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, h4.x + h4.y + h4.z + h4.w);
      if (lane == 0) s.wb[win] = sum;
    }
    if (tid == 0) s.pad_cnt = table[kRowsPadBin];
    row_sync();
    // ---- SCAN1b: every warp scans the window totals, high to low, then ranks
    // the bins of its own windows at or above the window holding the K-th
    // key: table[b] = above(b) | count(b) << 11 | log2ceil(count(b)) << 25.
    {
      const uint32_t wt = s.wb[kWindows - 1 - lane];  // lane l: window 31 - l
      const uint32_t wincl = warp_inclusive_scan(wt);
#pragma unroll
      for (int j = 0; j < kWindows / kWarpsT; ++j) {
        const int win = warp * (kWindows / kWarpsT) + j;
        const uint32_t above_w = __shfl_sync(0xFFFFFFFFu, wincl - wt, kWindows - 1 - win);
        const uint32_t tot_w = __shfl_sync(0xFFFFFFFFu, wt, kWindows - 1 - win);
        if (tot_w == 0u || above_w >= (uint32_t)ksel) continue;
        const int hi = 128 * win + 127;  // lane l: bins hi-4l .. hi-4l-3
        uint32_t h[4];
        load_bins_desc<4>(table + (hi - 4 * lane - 3), h);
        const uint32_t local = h[0] + h[1] + h[2] + h[3];
        const uint32_t incl = warp_inclusive_scan(local);
        uint32_t a = above_w + incl - local;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (h[e] != 0u && a < (uint32_t)ksel) {
            const int b = hi - 4 * lane - e;
            if ((uint32_t)ksel <= a + h[e]) {
              s.b1 = (uint32_t)b;
              s.nlive = a + h[e];
              s.above_b1 = a;
            }
            const uint32_t q = h[e] > 1u ? 32u - __clz(h[e] - 1u) : 0u;
            table[b] = a | (h[e] << 11) | (q << 25);
          }
          a += h[e];
        }
      }
    }
    row_sync();
    dbg_poison<NT>(s.wb, kMaxWarps);  // the window totals are dead

    // Live candidates are those with (key >> kRefShift) >= live_from: every
    // candidate of bins >= b1, unless that overflows the live list; then the
    // next 11 key bits of bin b1 are histogrammed (in `fine`, still zero) and
    // only its candidates from the digit holding the K-th key on stay live.
    const uint32_t b1 = s.b1;
    uint32_t live_from = b1 << 11;
    if (s.nlive > (uint32_t)kRowsLive) {
#pragma unroll
      for (int c = 0; c < kItems / 8; ++c) {
        uint32_t kc[8];
        tmem_load8(tkeys + 8 * c, kc);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = 8 * c + e;
          if ((tid + (j >> 2) * NT) < n4 && (kc[e] >> kL1Shift) == b1)
            atomicAdd(&s.fine[(kc[e] >> kRefShift) & 0x7FFu], 1u);
        }
      }
      row_sync();
      find_digit_desc<NT>(s.fine, (uint32_t)ksel - s.above_b1, s.wa, s.wb, s.found_digit,
                          s.found_above, s.found_count);
      row_sync();
      live_from |= s.found_digit;
      const uint32_t hb = s.found_above + s.found_count;  // live candidates of bin b1
      if constexpr (kPoisonBuild) {
        row_sync();
        dbg_poison<NT>(s.fine, kHistBins);
        __syncthreads();
      }
      zero_words<NT>(s.fine, kHistBins);
      row_sync();
      if (tid == 0) {
        s.nlive = s.above_b1 + hb;
        const uint32_t q = hb > 1u ? 32u - __clz(hb - 1u) : 0u;
        table[b1] = s.above_b1 | (hb << 11) | (q << 25);
      }
      row_sync();
    }
    const int nlive = (int)s.nlive;
    bool fast = nlive <= kRowsLive;
    const bool has_pad = s.pad_cnt != 0u;

    // ---- COMPACT: live candidates into a dense list ------------------------
    if (fast) {
      uint32_t mask = 0u;
      const uint32_t lf = live_from << kRefShift;  // live: key >= lf
      if (lf != 0u) {
        // candidates past the row hold key 0 (< lf)
#pragma unroll
        for (int c = 0; c < kItems / 8; ++c) {
          uint32_t kc[8];
          tmem_load8(tkeys + 8 * c, kc);
#pragma unroll
          for (int e = 0; e < 8; ++e) mask |= (kc[e] >= lf ? 1u : 0u) << (8 * c + e);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kItems; ++j) mask |= ((tid + (j >> 2) * NT) < n4 ? 1u : 0u) << j;
      }
      const uint32_t cnt = __popc(mask);
      const uint32_t incl = warp_inclusive_scan(cnt);
      uint32_t base = 0u;
      if (lane == 31) base = atomicAdd(&s.live_cursor, incl);
      unsigned long long* dst =
          s.live + dbg_clamp(__shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt, kRowsLive + 1u - cnt);
      // OR / AND of the row's inverted ids, taken as the AND / OR of the raw
      // ids.  Padding (a -inf key with the id -1) is left out of the OR: its
      // ~id of 0 is the smallest, so ordering on the varying bits alone still
      // puts it last.  Every other candidate counts, so a narrow row's
      // winners are their ~id bits under imask over the bits all of them
      // share (RANK rebuilds the ids that way).  The list holds the raw ids.
      uint32_t rand_ = 0xFFFFFFFFu, ror = 0u;  // AND / OR of the raw ids
      // the loop in two copies, with and without padding in the row
      auto compact_ids = [&](auto hp) {
        constexpr bool HP = decltype(hp)::value;
        uint32_t kc[8];  // the keys of chunks v and v+1, from tensor memory
#pragma unroll
      for (int v = 0; v < kVec; ++v) {
        if ((v & 1) == 0) tmem_load8(tkeys + 4 * v, kc);
        if ((tid + v * NT) < n4) {
          const uint4 iv = ivs[v];
          const uint32_t us[4] = {iv.x, iv.y, iv.z, iv.w};
          rand_ &= us[0] & us[1] & us[2] & us[3];
          if constexpr (HP) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              ror |= (us[e] == 0xFFFFFFFFu && kc[4 * (v & 1) + e] == kNegInfKey) ? 0u : us[e];
          }
          else
            ror |= us[0] | us[1] | us[2] | us[3];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (mask & (1u << (4 * v + e)))
              *dst++ = ((unsigned long long)kc[4 * (v & 1) + e] << 32) | us[e];
        }
      }
      };
      if (has_pad)
        compact_ids(std::true_type{});
      else
        compact_ids(std::false_type{});
      const uint32_t ior = ~__reduce_and_sync(0xFFFFFFFFu, rand_);
      const uint32_t iand = ~__reduce_or_sync(0xFFFFFFFFu, ror);
      if (lane == 0) {
        s.wior[warp] = ior;
        s.wiand[warp] = iand;
      }
    }
    row_sync();

    // ---- L2: the position-space bucket of every live candidate -------------
    // For finite scores the key bits below the L1 bin and below tzf are equal
    // within a sign, and the bits of ~id at or above ibf are equal for every
    // candidate of the row (but padding), so within one bin keys are ordered
    // like y = (low key bits >> tzf) << ibf | (~id low ibf bits), a wf-bit
    // number; its top q = log2ceil(count) bits, scaled onto the bin's count
    // buckets, name the bucket.  Bins up to kRowsPadBin (-inf, where padding
    // lives, and below) keep every bit.  Narrow rows (every live key above
    // that bin, wf <= 24) rank with 32-bit keys.
    const uint32_t ro = __reduce_or_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wraw[lane] : 0u);
    const uint32_t vi = __reduce_or_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wior[lane] : 0u) ^
                        __reduce_and_sync(0xFFFFFFFFu, lane < kWarpsT ? s.wiand[lane] : 0xFFFFFFFFu);
    const int tzf = ro ? min(__ffs(ro) - 1, kL1Shift) : kL1Shift;
    const int ibf = vi ? 32 - __clz(vi) : 0;
    const uint32_t imask = ibf >= 32 ? 0xFFFFFFFFu : ((1u << ibf) - 1u);
    const int wf = kL1Shift - tzf + ibf;
    const bool narrow = b1 > kRowsPadBin && wf <= 24;
    uint32_t gsl[kLivePer];  // wide rows: each list entry's bucket
    if (fast && narrow) {
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        const int e = tid + u * NT;
        if (e < nlive) {
          const unsigned long long lk = s.live[e];
          const uint32_t kk = (uint32_t)(lk >> 32);
          const uint32_t tb = table[kk >> kL1Shift];
          const int q = (int)(tb >> 25);
          const uint32_t y = (((kk & kLowMask) >> tzf) << ibf) | (~(uint32_t)lk & imask);
          const int d = wf - q;
          const uint32_t sub = d >= 0 ? (y >> d) : (y << (-d));
          const uint32_t cb = (tb >> 11) & 0x3FFFu;
          const uint32_t g = dbg_clamp((tb & 0x7FFu) + cb - 1u - ((sub * cb) >> q), kRowsFine);
          atomicAdd(&s.fine[g], 1u);
          // the entry becomes y << 32 | bin << 12 | bucket: SCATTER needs
          // nothing else, and no bucket ids wait in registers across SCAN2
          s.live[e] = ((unsigned long long)y << 32) | ((kk >> kL1Shift) << 12) | g;
        }
      }
    } else if (fast) {
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        const int e = tid + u * NT;
        gsl[u] = kNone;
        if (e < nlive) {
          const unsigned long long lk = s.live[e];
          const uint32_t kk = (uint32_t)(lk >> 32);
          const uint32_t inv = ~(uint32_t)lk;
          const uint32_t bin = kk >> kL1Shift;
          const uint32_t tb = table[bin];
          const int q = (int)(tb >> 25);
          unsigned long long y;
          int wy;
          if (bin > kRowsPadBin) {
            y = ((unsigned long long)((kk & kLowMask) >> tzf) << ibf) | (inv & imask);
            wy = wf;
          } else {
            y = ((unsigned long long)(kk & kLowMask) << 32) | inv;
            wy = kL1Shift + 32;
          }
          const uint32_t sub = wy >= q ? (uint32_t)(y >> (wy - q)) : (uint32_t)(y << (q - wy));
          const uint32_t cb = (tb >> 11) & 0x3FFFu;
          const uint32_t g = dbg_clamp((tb & 0x7FFu) + cb - 1u - ((sub * cb) >> q), kRowsFine);
          atomicAdd(&s.fine[g], 1u);
          gsl[u] = g;
        }
      }
    }
    row_sync();
    dbg_poison<NT>(s.region, kRowsRegionWords);  // the bin table is dead

    // ---- SCAN2: bucket starts over positions [0, nlive) ---------------------
    // fine[g] becomes start << 16 | size << 8, its low byte the fill cursor
    // for SCATTER.  A bucket of more than 255 keys (found in the first pass)
    // sends the row to the fallback, so the size byte never overflows on the
    // fast path.
    if (fast) {
      // warps whose buckets all lie past the last one only report a zero total
      const bool warp_busy = kFinePer * 32 * warp < nlive;
      static_assert(kFinePer % 2 == 0, "8-byte bucket pairs");
      uint32_t local = 0u, incl = 0u;
      uint32_t* my = s.fine + kFinePer * tid;
      if (warp_busy) {
        uint32_t orc = 0u;  // a bucket of more than 255 keys has a bit above 7
#pragma unroll
        for (int e = 0; e < kFinePer; e += 2) {
          const uint2 v2 = *reinterpret_cast<const uint2*>(my + e);
          local += v2.x + v2.y;
          orc |= v2.x | v2.y;
        }
        incl = warp_inclusive_scan(local);
        if (__any_sync(0xFFFFFFFFu, orc > kBigBucket) && lane == 0) s.overflow = 1u;
      }
      if (lane == 31) s.wa[warp] = incl;
      row_sync();
      if (warp_busy) {
        const uint32_t wt = lane < kWarpsT ? s.wa[lane] : 0u;
        const uint32_t wti = warp_inclusive_scan(wt);
        uint32_t st = __shfl_sync(0xFFFFFFFFu, wti - wt, warp) + incl - local;
        if (st < (uint32_t)ksel && (uint32_t)ksel <= st + local) {
          // this thread's buckets hold position K - 1: the end of its bucket
          uint32_t s0 = st;
          for (int e = 0; e < kFinePer; ++e) {
            const uint32_t c = my[e];
            if ((uint32_t)ksel <= s0 + c) {
              s.p_end = s0 + c;
              break;
            }
            s0 += c;
          }
        }
        // The sizes are read again rather than kept from the first pass: the
        // row's bucket ids (gsl) are live across this scan, and registers
        // are what limit four CTAs per SM.
        auto start = [&](uint32_t c) {
          const uint32_t w = (st << 16) | (c << 8);
          st += c;
          return w;
        };
#pragma unroll
        for (int e = 0; e < kFinePer; e += 2) {
          const uint2 v2 = *reinterpret_cast<const uint2*>(my + e);
          const uint32_t w0 = start(v2.x);
          const uint32_t w1 = start(v2.y);
          *reinterpret_cast<uint2*>(my + e) = make_uint2(w0, w1);
        }
      }
    }
    row_sync();
    fast = fast && s.overflow == 0u;

    // the next row into L2 now: it lands during SCATTER and RANK and stays
    // there until the next row's loads
    if (tid == 0 && t + G < T) src.prefetch_row(t + G);
    float* os = out_scores + (size_t)t * (size_t)K;
    int32_t* oi = out_ids + (size_t)t * (size_t)K;
    const uint32_t rbase = fast ? src.row_base(t) : 0u;
    if (fast && narrow) {
      // ---- SCATTER: rank key y << 8 | (255 - slot); members of a bucket
      // share y's top bits, so y orders them, identical keys by their slot.
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        const int e = tid + u * NT;
        if (e < nlive) {
          const unsigned long long ent = s.live[e];
          const uint32_t lo = (uint32_t)ent;
          const uint32_t old = atomicAdd(&s.fine[dbg_clamp(lo & 0xFFFu, kRowsFine)], 1u);
          if ((old >> 16) < (uint32_t)ksel) {
            const uint32_t pos = dbg_clamp((old >> 16) + (old & 0xFFu), kRowsRankMax);
            info32[pos] = (old & 0xFFFFu) | ((lo >> 12) << 16);
            rk32[pos] = ((uint32_t)(ent >> 32) << 8) | (255u - (old & 0xFFu));
          }
        }
      }
      row_sync();
      // ---- RANK: position = bucket start + members ranking above ---------
      const uint32_t p_end = min(s.p_end, (uint32_t)kRowsRankMax);
      // a winner's key and ~id from its bin and y: the key bits below tzf
      // are those of its sign (0 for positive scores, 1 for negative), the
      // ~id bits above ibf those every candidate but padding shares
      const uint32_t tzfill = (1u << tzf) - 1u;
      const uint32_t ihigh = __reduce_and_sync(
          0xFFFFFFFFu, lane < kWarpsT ? s.wiand[lane] : 0xFFFFFFFFu) & ~imask;
      // When every non-padding id is >= 0 (the usual case) their ~ids share
      // bit 31, no winner is id -1, and the output needs no test for it.
      auto rank_rows = [&](auto nonneg) {
        constexpr bool NONNEG = decltype(nonneg)::value;
#pragma unroll 2  // two positions per trip: measured 0.4% faster
      for (uint32_t p = tid; p < p_end; p += NT) {
        const uint32_t inf = info32[p];
        const uint32_t st = dbg_clamp(p - (inf & 0xFFu), p + 1u);
        const uint32_t cnt = dbg_clamp((inf >> 8) & 0xFFu, kRowsRankMax + 9u - st);
        const uint32_t mine = rk32[p];
        const uint32_t mc = __reduce_max_sync(__activemask(), cnt);
        uint32_t r = 0u;
        if (mc > 1u) {
          const uint32_t* b = rk32 + st;
          if (mc <= 4u) {
#pragma unroll
            for (uint32_t e = 0; e < 4u; ++e) r += (e < cnt && b[e] > mine) ? 1u : 0u;
          } else if (mc <= 8u) {
#pragma unroll
            for (uint32_t e = 0; e < 8u; ++e) r += (e < cnt && b[e] > mine) ? 1u : 0u;
          } else {
            for (uint32_t e = 0; e < cnt; ++e) r += b[e] > mine ? 1u : 0u;
          }
        }
        const uint32_t fin = st + r;
        if (fin < (uint32_t)ksel) {
          const uint32_t bin = inf >> 16;
          const uint32_t y = mine >> 8;
          const uint32_t kk = (bin << kL1Shift) | ((y >> ibf) << tzf) | (bin >= 0x800u ? 0u : tzfill);
          os[fin] = __uint_as_float(score_bits(kk));
          oi[fin] = NONNEG ? (int32_t)(rbase + ~((y & imask) | ihigh))
                          : src.out_id_from(rbase, (y & imask) | ihigh);
        }
      }
      };
      if (ihigh >> 31)
        rank_rows(std::true_type{});
      else
        rank_rows(std::false_type{});
    } else if (fast) {
      // ---- SCATTER: rank key (key without its L1 bin) << 12 | list index;
      // members of a bucket share their key's top 12 bits.
#pragma unroll
      for (int u = 0; u < kLivePer; ++u) {
        if (gsl[u] != kNone) {
          const uint32_t old = atomicAdd(&s.fine[gsl[u]], 1u);
          if ((old >> 16) < (uint32_t)ksel) {
            const uint32_t pos = dbg_clamp((old >> 16) + (old & 0xFFu), kRowsRankMax);
            const uint32_t e = (uint32_t)(tid + u * NT);
            info[pos] = (uint16_t)(old & 0xFFFFu);
            rk64[pos] = ((s.live[e] ^ 0xFFFFFFFFull) << 12) | e;
          }
        }
      }
      row_sync();
      // ---- RANK ----------------------------------------------------------
      const uint32_t p_end = min(s.p_end, (uint32_t)kRowsRankMax);
      for (uint32_t p = tid; p < p_end; p += NT) {
        const uint32_t inf = info[p];
        const uint32_t st = dbg_clamp(p - (inf & 0xFFu), p + 1u);
        const uint32_t cnt = dbg_clamp(inf >> 8, kRowsRankMax + 9u - st);
        const unsigned long long mine = rk64[p];
        const uint32_t mc = __reduce_max_sync(__activemask(), cnt);
        uint32_t r = 0u;
        if (mc > 1u) {
          const unsigned long long* b = rk64 + st;
          if (mc <= 4u) {
#pragma unroll
            for (uint32_t e = 0; e < 4u; ++e) r += (e < cnt && b[e] > mine) ? 1u : 0u;
          } else if (mc <= 8u) {
#pragma unroll
            for (uint32_t e = 0; e < 8u; ++e) r += (e < cnt && b[e] > mine) ? 1u : 0u;
          } else {
            for (uint32_t e = 0; e < cnt; ++e) r += b[e] > mine ? 1u : 0u;
          }
        }
        const uint32_t fin = st + r;
        if (fin < (uint32_t)ksel) {
          const unsigned long long key = s.live[dbg_clamp((uint32_t)mine & 0xFFFu, kRowsLive)];
          os[fin] = __uint_as_float(score_bits((uint32_t)(key >> 32)));
          oi[fin] = src.out_id_from(rbase, ~(uint32_t)key);
        }
      }
    } else {
      rows_fallback(src, s, t, n, os, oi);
    }
    row_sync();  // every reader of this row's shared state is done
    if constexpr (kPoisonBuild) {
      dbg_poison<NT>(s.fine, kRowsFine + kRowsRegionWords);
      dbg_poison<NT>(s.live, 2 * kRowsLive);
      dbg_poison<NT>(s.wa, 2 * kMaxWarps);
      if (tid == 0) {
        s.b1 = s.nlive = s.above_b1 = s.pad_cnt = s.pad_n = 0xA5A5A5A5u;
        s.found_digit = s.found_above = s.found_count = 0xA5A5A5A5u;
        s.live_cursor = s.p_end = s.overflow = 0xA5A5A5A5u;
        for (int w = 0; w < kWarpsT; ++w) s.wraw[w] = s.wior[w] = s.wiand[w] = 0xA5A5A5A5u;
      }
      __syncthreads();
    }
    zero_words<NT>(s.fine, kRowsFine + kRowsBins);  // fine and the histogram behind it
    if (tid == 0) {
      s.live_cursor = 0u;
      s.p_end = 0u;
      s.overflow = 0u;
    }
  }
  tmem_sync();  // every warp's last tensor-memory access is done
  if (warp == 0) tmem_dealloc64(s.tmem_base);
}

}  // namespace dcp
