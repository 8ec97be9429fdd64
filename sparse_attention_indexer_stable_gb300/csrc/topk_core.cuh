// topk_core.cuh -- general per-row stable top-K selection on sm_103a.
//
// One CTA of NT threads owns one query row at a time.  Given accessors for
// each candidate's 32-bit score key and inverted id, it
//   1. radix-selects the K-th largest score key with 11/11/10-bit digit
//      histograms ("[Kernel] Optimize CuTeDSL DCP top-k merge", Summary: a
//      radix pass over 32-bit score keys first),
//   2. only if that threshold is shared by more candidates than there are
//      slots left, radix-selects among the tied candidates on the inverted id
//      (same page: the token-id tie-break pass runs only when the score
//      threshold actually ties),
//   3. compacts the K winners as 64-bit keys score_key<<32 | ~id,
//   4. sorts them descending (score descending, then lowest id).
// This is the path for rows the streaming kernel (topk_fast.cuh) does not
// take, and its fallback for rows whose keys cluster too tightly.
//
// Barrier discipline: every phase that reads a shared result (threshold digit,
// counts) is separated by __syncthreads() from the next phase that resets or
// rewrites that shared state.  The review of the same page reports the bug
// this prevents: without a barrier between loading the threshold and zeroing
// it, late warps read 0 and drop every tied candidate.
#pragma once

#include <cstdint>

namespace dcp {

constexpr int kThreads = 1024;
constexpr int kMaxWarps = 32;
constexpr int kHistBins = 2048;

// Device status word: kernels set bits here on failures they detect (a
// staging copy that never completed, a misaligned shard, a clamped index in
// the race-check build); read and cleared by dcp_topk_device_status.
__device__ unsigned int g_device_status;
constexpr uint32_t kStatusPoisonClamp = 4u;  // race-check build: an index from shared state clamped

// ---- Race-check build (compiled with -DDCP_DEBUG_POISON) -------------------
// The race the first page's review reports: shared state reset while a late
// warp had not yet read it (a threshold loaded, then zeroed with no barrier
// in between; late warps read 0 and drop every tied candidate).  Whether such
// a missing barrier shows up depends on warp timing.  The race-check build
// removes the dependence:
//  - after every barrier of the row loops the odd warps wait a bounded while,
//    so at every phase boundary some warps are the late readers;
//  - every reset of shared state is preceded by an overwrite with garbage and
//    a barrier, so a reader that no barrier orders before the reset reads
//    garbage, not a value that might happen to be right;
//  - indices taken from shared state are clamped into their arrays and the
//    clamp recorded (kStatusPoisonClamp), so reading garbage cannot fault.
// A missing barrier then gives a wrong answer or a status bit, which the
// parity tests catch.  Without the macro all of this compiles to nothing.
#ifdef DCP_DEBUG_POISON
constexpr bool kPoisonBuild = true;
#else
constexpr bool kPoisonBuild = false;
#endif

// Race-check build: the odd warps wait about 3000 cycles (a bounded delay).
__device__ __forceinline__ void dbg_skew() {
  if constexpr (kPoisonBuild) {
    if ((threadIdx.x >> 5) & 1u) {
      const long long t0 = clock64();
      while (clock64() - t0 < 3000) {
      }
    }
  }
}

// __syncthreads(), then the race-check build's skew.
__device__ __forceinline__ void row_sync() {
  __syncthreads();
  dbg_skew();
}

// Race-check build: `words` 32-bit words at p overwritten with garbage by
// the CTA's NT threads.
template <int NT>
__device__ __forceinline__ void dbg_poison(void* p, int words) {
  if constexpr (kPoisonBuild) {
    uint32_t* w = reinterpret_cast<uint32_t*>(p);
    for (int i = threadIdx.x; i < words; i += NT) w[i] = 0xA5A5A5A5u ^ ((uint32_t)i * 0x9E3779B9u);
  }
}

// Race-check build: i clamped into [0, n), the clamp recorded.
__device__ __forceinline__ uint32_t dbg_clamp(uint32_t i, uint32_t n) {
  if constexpr (kPoisonBuild) {
    if (i >= n) {
      atomicOr(&g_device_status, kStatusPoisonClamp);
      return n - 1u;
    }
  }
  return i;
}

// Order-preserving map of fp32 bits to u32: unsigned order of the result is
// float order, with -0.0 just below +0.0 and NaNs outside the finite range.
// Negative values have every bit inverted, the others only the sign bit.
__device__ __forceinline__ uint32_t score_key(uint32_t bits) {
  return bits ^ ((uint32_t)((int32_t)bits >> 31) | 0x80000000u);
}

// Inverse of score_key: the original fp32 bits.
__device__ __forceinline__ uint32_t score_bits(uint32_t key) {
  return key ^ ((uint32_t)((int32_t)~key >> 31) | 0x80000000u);
}

struct SelectShared {
  uint32_t hist[kHistBins];
  uint32_t warp_sum[kMaxWarps];
  uint32_t warp_off[kMaxWarps];
  uint32_t found_digit;
  uint32_t found_above;
  uint32_t found_count;
  uint32_t win_count;
  uint32_t dup_claim;
};

// Inclusive prefix sum across the warp (all 32 lanes active).  The shuffle's
// predicate says whether the source lane exists, so each step is a shuffle
// and a predicated add.
__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    asm("{\n .reg .u32 t;\n .reg .pred p;\n"
        " shfl.sync.up.b32 t|p, %0, %1, 0, 0xffffffff;\n"
        " @p add.u32 %0, %0, t;\n}\n"
        : "+r"(v)
        : "r"(o));
  }
  return v;
}

// Finds the digit d of the histogram with above(d) < need <= above(d) + hist[d],
// above(d) = sum of hist[e] for e > d; nbins <= 2048.  Exactly one thread
// writes found_*; the caller must __syncthreads() before reading them.
template <int NT>
__device__ __forceinline__ void find_threshold_digit(SelectShared& s, int nbins, uint32_t need) {
  constexpr int kPer = kHistBins / NT;  // bins per thread, descending
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t h[kPer];
  uint32_t local = 0u;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int b = nbins - 1 - (kPer * tid + e);
    h[e] = b >= 0 ? s.hist[b] : 0u;
    local += h[e];
  }
  const uint32_t incl = warp_inclusive_scan(local);
  if (lane == 31) s.warp_sum[warp] = incl;
  row_sync();
  if (warp == 0) {
    const uint32_t w = lane < NT / 32 ? s.warp_sum[lane] : 0u;
    const uint32_t wi = warp_inclusive_scan(w);
    s.warp_off[lane] = wi - w;
  }
  row_sync();
  uint32_t above = s.warp_off[warp] + incl - local;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    if (h[e] != 0u && above < need && need <= above + h[e]) {
      s.found_digit = (uint32_t)(nbins - 1 - (kPer * tid + e));
      s.found_above = above;
      s.found_count = h[e];
    }
    above += h[e];
  }
}

// Result of a radix select over one 32-bit value per participating candidate.
// The selected ones are those with (v & mask) > prefix, plus `need` of those
// with (v & mask) == prefix (which number `count`).  If need == count they all
// are; otherwise mask == ~0u and the `count` candidates are exact duplicates
// of the value `prefix`.
struct RadixResult {
  uint32_t mask;
  uint32_t prefix;
  uint32_t need;
  uint32_t count;
};

// Radix select of the `need` largest values (1 <= need <= participants).
// ValueFn(i, v) -> bool: whether candidate i participates, and its value.
template <int NT, class ValueFn>
__device__ __forceinline__ RadixResult radix_select(SelectShared& s, int n, uint32_t need,
                                                    ValueFn value) {
  const int tid = threadIdx.x;
  RadixResult r{0u, 0u, need, 0u};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nbins = pass == 2 ? 1024 : 2048;
    const uint32_t dmask = (uint32_t)nbins - 1u;
    if constexpr (kPoisonBuild) {
      dbg_poison<NT>(&s, (int)(sizeof(SelectShared) / 4));
      __syncthreads();
    }
    for (int b = tid; b < nbins; b += NT) s.hist[b] = 0u;
    row_sync();
    for (int i = tid; i < n; i += NT) {
      uint32_t v;
      if (value(i, v) && (v & r.mask) == r.prefix) atomicAdd(&s.hist[(v >> shift) & dmask], 1u);
    }
    row_sync();
    find_threshold_digit<NT>(s, nbins, r.need);
    row_sync();
    const uint32_t d = s.found_digit, above = s.found_above, cnt = s.found_count;
    r.need -= above;
    r.prefix |= d << shift;
    r.mask |= dmask << shift;
    r.count = cnt;
    // Every thread has now read found_* and the histogram; only after this
    // barrier may the next pass (or the caller) reset them.
    row_sync();
    if (cnt == r.need) break;
  }
  return r;
}

// Bitonic sort of n_pow2 64-bit keys in shared memory, descending.
template <int NT>
__device__ __forceinline__ void bitonic_sort_desc(unsigned long long* a, int n_pow2) {
  const int tid = threadIdx.x;
  for (int k = 2; k <= n_pow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < (n_pow2 >> 1); i += NT) {
        const int lo = 2 * i - (i & (j - 1));
        const int hi = lo + j;
        const unsigned long long x = a[lo], y = a[hi];
        const bool desc = (lo & k) == 0;
        if (desc ? (x < y) : (x > y)) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      row_sync();
    }
  }
}

// The whole per-row selection over n candidates given by accessors:
// key(i) -> 32-bit score key, inv(i) -> inverted id.  On return
// win[0..ksel) holds the winners sorted descending by 64-bit key.
// n_pow2: a power of two >= ksel; win must have room for n_pow2 keys.
template <int NT, class KeyFn, class InvFn>
__device__ __forceinline__ void select_sort_row(SelectShared& s, int n, int ksel,
                                                unsigned long long* win, int n_pow2,
                                                KeyFn key, InvFn inv) {
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  // 1. Threshold on the 32-bit score key.
  const RadixResult rs = radix_select<NT>(s, n, (uint32_t)ksel, [&](int i, uint32_t& v) {
    v = key(i);
    return true;
  });

  // 2. Tie-break on the inverted id, only when the threshold key ties beyond
  //    the remaining slots.
  const bool tie = rs.need != rs.count;
  RadixResult rt{0u, 0u, 0u, 0u};
  if (tie) {
    const uint32_t tau = rs.prefix;
    rt = radix_select<NT>(s, n, rs.need, [&](int i, uint32_t& v) {
      v = inv(i);
      return key(i) == tau;
    });
  }
  const bool dup = tie && rt.need != rt.count;
  if (tid == 0) {
    s.win_count = 0u;
    s.dup_claim = 0u;
  }
  row_sync();

  // 3. Compaction of the winners (order is irrelevant: the sort below fixes
  //    it, and candidates with equal 64-bit keys are identical).
  for (int base = 0; base < n; base += NT) {
    const int i = base + tid;
    bool w = false;
    uint32_t k = 0u, u = 0u;
    if (i < n) {
      k = key(i);
      u = inv(i);
      const uint32_t km = k & rs.mask;
      if (km > rs.prefix) {
        w = true;
      } else if (km == rs.prefix) {
        if (!tie) {
          w = true;
        } else {
          const uint32_t um = u & rt.mask;
          if (um > rt.prefix) w = true;
          else if (um == rt.prefix) w = !dup || atomicAdd(&s.dup_claim, 1u) < rt.need;
        }
      }
    }
    const uint32_t ballot = __ballot_sync(0xFFFFFFFFu, w);
    uint32_t slot0 = 0u;
    if (lane == 0 && ballot) slot0 = atomicAdd(&s.win_count, (uint32_t)__popc(ballot));
    slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
    if (w) {
      const uint32_t slot = slot0 + (uint32_t)__popc(ballot & ((1u << lane) - 1u));
      if (slot < (uint32_t)n_pow2) win[slot] = ((unsigned long long)k << 32) | u;
    }
  }
  for (int j = ksel + tid; j < n_pow2; j += NT) win[j] = 0ull;
  row_sync();

  // 4. Final order.
  bitonic_sort_desc<NT>(win, n_pow2);
}

}  // namespace dcp
