// dcp_topk.cu -- kernels and C ABI of the DCP top-K library (sm_103a).
//
// Entry points are declared and documented in include/dcp_topk.h.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "dcp_topk.h"
#include "topk_core.cuh"
#include "topk_fast.cuh"
#include "topk_rows.cuh"

namespace dcp {

// Rows are walked 1024 at a time, as the merge of "Reserve the sparse
// indexer's DCP top-k merge scratch through the workspace manager" (Purpose)
// does; rows are independent, so this only fixes the order of the walk.
constexpr int kChunkRows = 1024;

// The candidates of a merge.  Shard r's row t holds K scores and K ids:
// - rank-major layout (Indirect = false): one (dcp, T, K) buffer each, shard
//   r of row t at (r*T + t)*K, as the gather of "Reserve the sparse indexer's
//   DCP top-k merge scratch through the workspace manager" (Purpose) leaves
//   them;
// - separate shards (Indirect = true): a device array of dcp pointers to
//   (T, K) row-major shards, row t of shard r at shard[r] + t*K, the shards
//   read where they lie ("[DCP][Performance] Add Shared-DCP peer-addressable
//   decode data paths", Summary: the Top-K consumer reads owner-local and
//   peer shards through views instead of an inbox).
// Candidate index i = r*K + k in both.
template <bool Indirect>
struct MergeSourceT {
  const float* scores;               // rank-major layout
  const int32_t* ids;
  const float* const* shard_scores;  // separate shards: device arrays of dcp pointers
  const int32_t* const* shard_ids;
  const int32_t* row_starts;
  int T, dcp, K;
  bool vec4;
  static constexpr bool kIndirect = Indirect;
  static constexpr bool kMerge = true;

  // Row t of shard r.
  __device__ const float* score_row(int t, int r) const {
    if constexpr (Indirect)
      return reinterpret_cast<const float*>(
                 __ldg(reinterpret_cast<const unsigned long long*>(shard_scores) + r)) +
             (size_t)t * (size_t)K;
    else
      return scores + ((size_t)r * T + t) * (size_t)K;
  }
  __device__ const int32_t* id_row(int t, int r) const {
    if constexpr (Indirect)
      return reinterpret_cast<const int32_t*>(
                 __ldg(reinterpret_cast<const unsigned long long*>(shard_ids) + r)) +
             (size_t)t * (size_t)K;
    else
      return ids + ((size_t)r * T + t) * (size_t)K;
  }
  // Whether every shard pointer allows the 16-byte copies of the fast paths
  // (separate shards: the host cannot see the device-resident pointers).
  __device__ bool shards_aligned() const {
    if constexpr (Indirect) {
      uintptr_t bits = 0;
      for (int r = 0; r < dcp; ++r)
        bits |= (uintptr_t)score_row(0, r) | (uintptr_t)id_row(0, r);
      return (bits & 15u) == 0;
    } else {
      return true;
    }
  }

  __device__ int count() const { return dcp * K; }

  // Candidates of row t: index i = r*K + k.
  __device__ void stage(int t, uint32_t* skey, uint32_t* sinv) const {
    const int n = dcp * K;
    if (vec4) {
      const int k4 = K >> 2;
      for (int q = threadIdx.x; q < (n >> 2); q += kThreads) {
        const int r = q / k4;
        const int kk = (q - r * k4) << 2;
        const uint4 sb = __ldg(reinterpret_cast<const uint4*>(score_row(t, r) + kk));
        const int4 ib = __ldg(reinterpret_cast<const int4*>(id_row(t, r) + kk));
        const int i = r * K + kk;
        *reinterpret_cast<uint4*>(skey + i) =
            make_uint4(score_key(sb.x), score_key(sb.y), score_key(sb.z), score_key(sb.w));
        *reinterpret_cast<uint4*>(sinv + i) =
            make_uint4(~(uint32_t)ib.x, ~(uint32_t)ib.y, ~(uint32_t)ib.z, ~(uint32_t)ib.w);
      }
    } else {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int r = i / K;
        const int k = i - r * K;
        skey[i] = score_key(__float_as_uint(__ldg(score_row(t, r) + k)));
        sinv[i] = ~(uint32_t)__ldg(id_row(t, r) + k);
      }
    }
  }

  // Fast path staging: the row's scores and its ids, each as dcp 16-byte
  // copies straight from the shards (needs K % 4 == 0 and 16-byte aligned
  // shards), completing on separate barriers.
  static constexpr bool kStagesIds = true;
  // ids are arbitrary: their order is not the candidates' order
  __device__ bool index_ordered() const { return false; }
  __host__ __device__ int score_words() const { return dcp * K; }
  __host__ __device__ int ids_words() const { return dcp * K; }

  // One thread: arm `bar` with the bytes of row t's scores and copy them to dst.
  __device__ void issue_scores(int t, uint32_t* dst, unsigned long long* bar) const {
    const uint32_t seg = (uint32_t)K * 4u;
    mbar_expect_tx(bar, (uint32_t)dcp * seg);
    for (int r = 0; r < dcp; ++r) tma_load_1d(dst + r * K, score_row(t, r), seg, bar);
  }

  // One thread: the same for row t's ids.
  __device__ void issue_ids(int t, uint32_t* dst, unsigned long long* bar) const {
    const uint32_t seg = (uint32_t)K * 4u;
    mbar_expect_tx(bar, (uint32_t)dcp * seg);
    for (int r = 0; r < dcp; ++r) tma_load_1d(dst + r * K, id_row(t, r), seg, bar);
  }

  // Inverted ids of staged candidates 4c .. 4c+3 (staged ids at `staged`).
  __device__ uint4 inv4(const uint32_t* staged, int c) const {
    const uint4 w = *reinterpret_cast<const uint4*>(staged + 4 * c);
    return make_uint4(~w.x, ~w.y, ~w.z, ~w.w);
  }

  // Candidate i of row t read from global memory (the fallback path).
  __device__ uint32_t key_global(int t, int i) const {
    const int r = i / K;
    return score_key(__float_as_uint(__ldg(score_row(t, r) + (i - r * K))));
  }
  __device__ uint32_t inv_global(int t, int i) const {
    const int r = i / K;
    return ~(uint32_t)__ldg(id_row(t, r) + (i - r * K));
  }
  // Score keys of candidates 4c .. 4c+3 of row t (one shard: K % 4 == 0).
  __device__ uint4 key4_global(int t, int c) const {
    const int i = 4 * c, r = i / K;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(score_row(t, r) + (i - r * K)));
    return make_uint4(score_key(w.x), score_key(w.y), score_key(w.z), score_key(w.w));
  }

  // Ids of candidates 4c .. 4c+3 of row t (one shard: K % 4 == 0).
  __device__ uint4 ids4_global(int t, int c) const {
    const int i = 4 * c, r = i / K;
    return __ldg(reinterpret_cast<const uint4*>(id_row(t, r) + (i - r * K)));
  }

  // One thread: pulls row t's scores and ids of every shard into L2.
  __device__ void prefetch_row(int t) const {
    for (int r = 0; r < dcp; ++r) {
      prefetch_l2(score_row(t, r), (uint32_t)K * 4u);
      prefetch_l2(id_row(t, r), (uint32_t)K * 4u);
    }
  }

  // Per-row part of the output id, read once per row.
  __device__ uint32_t row_base(int t) const {
    return row_starts ? (uint32_t)__ldg(row_starts + t) : 0u;
  }

  __device__ int32_t out_id_from(uint32_t base, uint32_t inv) const {
    const uint32_t id = ~inv;
    return id == 0xFFFFFFFFu ? -1 : (int32_t)(id + base);
  }

  __device__ int32_t out_id(int t, uint32_t inv) const {
    const uint32_t id = ~inv;
    if (id == 0xFFFFFFFFu) return -1;
    const uint32_t rs = row_starts ? (uint32_t)__ldg(row_starts + t) : 0u;
    return (int32_t)(id + rs);
  }
};
using MergeSource = MergeSourceT<false>;
using ShardsSource = MergeSourceT<true>;

// Column c of one rank's shard is candidate c (ordered by ~c: the global id
// grows with the column in both shard layouts); its global id is
// row_starts[t] + id_offset + c*id_stride.
struct LocalSource {
  const float* logits;
  const int32_t* row_starts;
  int L, ld, rank;
  bool vec4;
  uint32_t id_offset;  // rank*L (contiguous shards) or rank (interleaved)
  uint32_t id_stride;  // 1 (contiguous) or dcp (interleaved)

  __device__ int count() const { return L; }

  __device__ void stage(int t, uint32_t* skey, uint32_t* sinv) const {
    const float* row = logits + (size_t)t * (size_t)ld;
    if (vec4) {
      for (int q = threadIdx.x; q < (L >> 2); q += kThreads) {
        const uint4 sb = __ldg(reinterpret_cast<const uint4*>(row) + q);
        const int c = q << 2;
        *reinterpret_cast<uint4*>(skey + c) =
            make_uint4(score_key(sb.x), score_key(sb.y), score_key(sb.z), score_key(sb.w));
        *reinterpret_cast<uint4*>(sinv + c) =
            make_uint4(~(uint32_t)c, ~(uint32_t)(c + 1), ~(uint32_t)(c + 2), ~(uint32_t)(c + 3));
      }
    } else {
      for (int c = threadIdx.x; c < L; c += kThreads) {
        skey[c] = score_key(__float_as_uint(__ldg(row + c)));
        sinv[c] = ~(uint32_t)c;
      }
    }
  }

  // Ids are column numbers: only the logits are staged.
  static constexpr bool kStagesIds = false;
  static constexpr bool kIndirect = false;
  static constexpr bool kMerge = false;
  __device__ bool shards_aligned() const { return true; }
  __device__ bool index_ordered() const { return true; }  // ids grow with the column
  __host__ __device__ int score_words() const { return L; }
  __host__ __device__ int ids_words() const { return 0; }

  __device__ void issue_scores(int t, uint32_t* dst, unsigned long long* bar) const {
    mbar_expect_tx(bar, (uint32_t)L * 4u);
    tma_load_1d(dst, logits + (size_t)t * (size_t)ld, (uint32_t)L * 4u, bar);
  }
  __device__ void issue_ids(int, uint32_t*, unsigned long long*) const {}

  __device__ uint4 inv4(const uint32_t*, int c) const {
    const uint32_t i = 4u * (uint32_t)c;
    return make_uint4(~i, ~(i + 1u), ~(i + 2u), ~(i + 3u));
  }

  __device__ uint32_t row_base(int t) const {
    return (row_starts ? (uint32_t)__ldg(row_starts + t) : 0u) + id_offset;
  }


  __device__ uint32_t key_global(int t, int i) const {
    return score_key(__float_as_uint(__ldg(logits + (size_t)t * (size_t)ld + i)));
  }
  __device__ uint32_t inv_global(int, int i) const { return ~(uint32_t)i; }

  __device__ int32_t out_id_from(uint32_t base, uint32_t inv) const {
    return (int32_t)(base + ~inv * id_stride);
  }

  __device__ int32_t out_id(int t, uint32_t inv) const { return out_id_from(row_base(t), inv); }
};

// All dcp shards' logits of a row at once: candidate i = r*L + c is column c
// of shard r's row (logits rank-major (dcp, T, ld)), global id
// row_starts[t] + r*L + c.  By the composition of the local top-K and the
// merge, the result equals merging the shards' local top-K.
struct FusedSource {
  const float* logits;
  const int32_t* row_starts;
  int T, dcp, L, ld;
  bool vec4;
  bool interleaved;             // ids c*dcp + r instead of r*L + c
  unsigned long long l_recip;   // ceil(2^32 / L): r = (i * l_recip) >> 32 for i < dcp*L

  // Global id (before row_starts) of candidate i = r*L + c.  The quotient by
  // multiplication is exact because i*L < 2^32.
  __device__ uint32_t gid(uint32_t i) const {
    if (!interleaved) return i;
    const uint32_t r = (uint32_t)(((unsigned long long)i * l_recip) >> 32);
    return (i - r * (uint32_t)L) * (uint32_t)dcp + r;
  }

  __device__ int count() const { return dcp * L; }

  __device__ const float* row(int t, int r) const {
    return logits + ((size_t)r * T + t) * (size_t)ld;
  }

  __device__ void stage(int t, uint32_t* skey, uint32_t* sinv) const {
    for (int r = 0; r < dcp; ++r) {
      const float* rp = row(t, r);
      for (int c = threadIdx.x; c < L; c += kThreads) {
        skey[r * L + c] = score_key(__float_as_uint(__ldg(rp + c)));
        sinv[r * L + c] = ~gid((uint32_t)(r * L + c));
      }
    }
  }

  // Ids are r*L + c: only the logits are staged.
  static constexpr bool kStagesIds = false;
  static constexpr bool kIndirect = false;
  static constexpr bool kMerge = false;
  __device__ bool shards_aligned() const { return true; }
  // ids grow with the candidate index only in the contiguous layout
  __device__ bool index_ordered() const { return !interleaved; }
  __host__ __device__ int score_words() const { return dcp * L; }
  __host__ __device__ int ids_words() const { return 0; }

  __device__ void issue_scores(int t, uint32_t* dst, unsigned long long* bar) const {
    const uint32_t seg = (uint32_t)L * 4u;
    mbar_expect_tx(bar, (uint32_t)dcp * seg);
    for (int r = 0; r < dcp; ++r) tma_load_1d(dst + r * L, row(t, r), seg, bar);
  }
  __device__ void issue_ids(int, uint32_t*, unsigned long long*) const {}

  // Candidates 4c .. 4c+3 lie in one shard (L % 4 == 0 on this path).
  __device__ uint4 inv4(const uint32_t*, int c) const {
    const uint32_t g = gid(4u * (uint32_t)c);
    const uint32_t d = interleaved ? (uint32_t)dcp : 1u;
    return make_uint4(~g, ~(g + d), ~(g + 2u * d), ~(g + 3u * d));
  }

  __device__ uint32_t row_base(int t) const {
    return row_starts ? (uint32_t)__ldg(row_starts + t) : 0u;
  }


  __device__ uint32_t key_global(int t, int i) const {
    const int r = i / L;
    return score_key(__float_as_uint(__ldg(row(t, r) + (i - r * L))));
  }
  __device__ uint32_t inv_global(int, int i) const { return ~gid((uint32_t)i); }

  __device__ int32_t out_id_from(uint32_t base, uint32_t inv) const {
    return (int32_t)(base + ~inv);
  }

  __device__ int32_t out_id(int t, uint32_t inv) const { return out_id_from(row_base(t), inv); }
};

__host__ __device__ inline int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Dynamic shared memory: SelectShared | win[n_pow2] (u64) | skey[n] | sinv[n],
// each part 16-byte aligned.
__host__ __device__ inline size_t row_smem_bytes(int n, int k) {
  const int ksel = k < n ? k : n;
  return align16(sizeof(SelectShared)) + align16((size_t)next_pow2(ksel) * 8) +
         2 * align16((size_t)n * 4);
}

template <class Source>
__global__ void __launch_bounds__(kThreads, 1)
    topk_rows_kernel(Source src, int T, int K, float* __restrict__ out_scores,
                     int32_t* __restrict__ out_ids) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SelectShared& s = *reinterpret_cast<SelectShared*>(smem_raw);
  const int n = src.count();
  const int ksel = K < n ? K : n;
  const int n_pow2 = next_pow2(ksel);
  unsigned char* p = smem_raw + align16(sizeof(SelectShared));
  unsigned long long* win = reinterpret_cast<unsigned long long*>(p);
  p += align16((size_t)n_pow2 * 8);
  uint32_t* skey = reinterpret_cast<uint32_t*>(p);
  p += align16((size_t)n * 4);
  uint32_t* sinv = reinterpret_cast<uint32_t*>(p);

  grid_dependency_wait();
  const int grid = (int)gridDim.x;
  const int b = (int)blockIdx.x;
  for (int cs = 0; cs < T; cs += kChunkRows) {
    const int ce = min(T, cs + kChunkRows);
    // first row of this chunk owned by this CTA: t == b (mod grid)
    int t = cs + (((b - cs) % grid) + grid) % grid;
    for (; t < ce; t += grid) {
      src.stage(t, skey, sinv);
      row_sync();
      select_sort_row<kThreads>(s, n, ksel, win, n_pow2, [&](int i) { return skey[i]; },
                                [&](int i) { return sinv[i]; });
      float* os = out_scores + (size_t)t * (size_t)K;
      int32_t* oi = out_ids + (size_t)t * (size_t)K;
      for (int j = threadIdx.x; j < K; j += kThreads) {
        if (j < ksel) {
          const unsigned long long w = win[j];
          os[j] = __uint_as_float(score_bits((uint32_t)(w >> 32)));
          oi[j] = src.out_id(t, (uint32_t)w);
        } else {
          os[j] = __uint_as_float(0xFF800000u);  // -inf
          oi[j] = -1;
        }
      }
      // The next row's staging overwrites skey/sinv/win.
      row_sync();
      if constexpr (kPoisonBuild) {
        dbg_poison<kThreads>(smem_raw, (int)(row_smem_bytes(n, K) / 4));
        __syncthreads();
      }
    }
  }
}


static cudaError_t status_word(unsigned int** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_device_status);
}

struct DeviceInfo {
  int sms = 0;
  int max_smem_optin = 0;
  unsigned int* status = nullptr;  // device address of g_device_status
  std::atomic<bool> configured{false};
};

static DeviceInfo g_dev[64];
static std::mutex g_dev_mutex;

template <class K>
static cudaError_t allow_max_smem(K kernel, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

// The streaming kernel's instantiations for one source: 512-thread CTAs two
// per SM, 1024-thread CTAs one per row, 1024-thread CTAs for rows of up to
// 16384 candidates, and the same for K up to 4096.
template <class Source>
static cudaError_t allow_stream_kernels(int smem) {
  cudaError_t e;
  if ((e = allow_max_smem(topk_stream_kernel<512, kStreamMaxN, kStreamMaxK, Source, false>,
                          smem)) != cudaSuccess)
    return e;
  if ((e = allow_max_smem(topk_stream_kernel<1024, kStreamMaxN, kStreamMaxK, Source, true>,
                          smem)) != cudaSuccess)
    return e;
  if ((e = allow_max_smem(topk_stream_kernel<1024, kStreamMaxNWide, kStreamMaxK, Source, true>,
                          smem)) != cudaSuccess)
    return e;
  return allow_max_smem(
      topk_stream_kernel<1024, kStreamMaxNWide, kStreamMaxKWide, Source, true>, smem);
}

// Per-device launch limits and kernel attributes, set once per device (the
// first call on a device must therefore not be inside a stream capture).
static cudaError_t device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  DeviceInfo& d = g_dev[dev];
  if (d.configured.load(std::memory_order_acquire)) {
    *out = &d;
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!d.configured.load(std::memory_order_relaxed)) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const int smem = d.max_smem_optin;
    if ((e = allow_max_smem(topk_rows_kernel<MergeSource>, smem)) != cudaSuccess) return e;
    if ((e = allow_max_smem(topk_rows_kernel<ShardsSource>, smem)) != cudaSuccess) return e;
    if ((e = allow_max_smem(topk_rows_kernel<LocalSource>, smem)) != cudaSuccess) return e;
    if ((e = allow_max_smem(topk_rows_kernel<FusedSource>, smem)) != cudaSuccess) return e;
    if ((e = allow_stream_kernels<MergeSource>(smem)) != cudaSuccess) return e;
    if ((e = allow_stream_kernels<ShardsSource>(smem)) != cudaSuccess) return e;
    if ((e = allow_stream_kernels<LocalSource>(smem)) != cudaSuccess) return e;
    if ((e = allow_stream_kernels<FusedSource>(smem)) != cudaSuccess) return e;
    if ((e = allow_max_smem(merge_rows_kernel<MergeSource>, (int)sizeof(RowsShared))) !=
        cudaSuccess)
      return e;
    if ((e = allow_max_smem(merge_rows_kernel<ShardsSource>, (int)sizeof(RowsShared))) !=
        cudaSuccess)
      return e;
    if ((e = status_word(&d.status)) != cudaSuccess) return e;
    d.configured.store(true, std::memory_order_release);
  }
  *out = &d;
  return cudaSuccess;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Launches with programmatic stream serialization: the grid may be scheduled
// while the stream's previous kernel is still finishing, and waits for it
// (griddepcontrol.wait, in every thread before its first global memory
// access) before touching memory.  Only the launch latency and shared-memory
// set-up overlap; the ordering is the stream's.
template <typename... KArgs, typename... Args>
static cudaError_t launch_serialized(void (*kernel)(KArgs...), dim3 grid, int block, size_t smem,
                                     cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// A kernel whose row copy is armed but never issued: exercises the bounded
// wait and the status report.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit, unsigned int* status) {
  __shared__ unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1u);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_expect_tx(&bar, 16u);
  const bool ok = mbar_wait_bounded(&bar, 0u, limit);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicOr(status, kStatusCopyTimeout);
}

// The many-row merge at K = 2048 (more than two rows per SM, dcp <= 4,
// 16-byte aligned rows): four 256-thread CTAs per SM walking the rows.  Otherwise the
// streaming path when the row fits it (n <= 16384, K <= 4096, 16-byte copies
// possible): one 1024-thread CTA per row when the rows fit on the SMs at
// once, else two 512-thread CTAs per SM walking the rows.  The general path
// otherwise.
template <class Source>
static dcp_status launch_rows(const Source& src, int T, int n, int K, float* out_scores,
                              int32_t* out_ids, cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  if (device_info(&d) != cudaSuccess) return DCP_ERR_CUDA;
  // The streaming kernel when 16-byte copies are possible and the row fits
  // it: two 512-thread CTAs per SM walking many rows of up to 8192
  // candidates; else one 1024-thread CTA per row (few rows, up to 16384
  // candidates, or K up to 4096).
  const bool big_k = K > kStreamMaxK;
  const bool two_per_sm = T > d->sms && n <= kStreamMaxN && !big_k;
  const size_t smem =
      big_k ? stream_smem_bytes<1024, kStreamMaxKWide>(src.score_words(), src.ids_words())
      : two_per_sm ? stream_smem_bytes<512>(src.score_words(), src.ids_words())
                   : stream_smem_bytes<1024>(src.score_words(), src.ids_words());
  const bool stream_ok = src.vec4 && K <= kStreamMaxKWide && n <= kStreamMaxNWide &&
                         smem <= (size_t)d->max_smem_optin;
  const int grid1 = T < d->sms ? T : d->sms;
  // Few rows: each row's sort split over up to 8 CTAs (parts, the grid's y
  // dimension), every part selecting the whole row's threshold and sorting a
  // slice of at least 256 of its min(K, n) winners, while the parts fit on
  // the SMs at once.
  const int ksel = K < n ? K : n;
  int parts = T > 0 ? d->sms / T : 1;
  parts = parts < 8 ? parts : 8;
  parts = parts < ksel / 256 ? parts : ksel / 256;
  parts = parts > 1 ? parts : 1;
  const dim3 gridp((unsigned)grid1, (unsigned)parts);  // T * parts <= sms when parts > 1
  const int slice = ksel / parts;
  cudaError_t e;
  if constexpr (Source::kMerge) {
    // above two rows per SM (at or below, the streaming kernel's two
    // 512-thread CTAs per SM measured faster: 256 rows 11.5 vs 12.2 us)
    if (src.vec4 && K == kRowsK && n <= kRowsMaxN && T > 2 * d->sms &&
        sizeof(RowsShared) <= (size_t)d->max_smem_optin) {
      const int grid = T < 4 * d->sms ? T : 4 * d->sms;
      e = launch_serialized(merge_rows_kernel<Source>, grid, kRowsNT, sizeof(RowsShared), stream,
                            src, T, out_scores, out_ids, d->status);
      return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
    }
  }
  if (stream_ok && big_k) {
    e = launch_serialized(
        topk_stream_kernel<1024, kStreamMaxNWide, kStreamMaxKWide, Source, true>, gridp, 1024,
        smem, stream, src, T, K, slice, out_scores, out_ids, d->status);
  } else if (stream_ok && n > kStreamMaxN) {
    e = launch_serialized(topk_stream_kernel<1024, kStreamMaxNWide, kStreamMaxK, Source, true>,
                          gridp, 1024, smem, stream, src, T, K, slice, out_scores, out_ids,
                          d->status);
  } else if (stream_ok && !two_per_sm) {
    e = launch_serialized(topk_stream_kernel<1024, kStreamMaxN, kStreamMaxK, Source, true>, gridp,
                          1024, smem, stream, src, T, K, slice, out_scores, out_ids, d->status);
  } else if (stream_ok) {
    const int grid = T < 2 * d->sms ? T : 2 * d->sms;
    e = launch_serialized(topk_stream_kernel<512, kStreamMaxN, kStreamMaxK, Source, false>, grid,
                          512, smem, stream, src, T, K, 1, out_scores, out_ids, d->status);
  } else {
    const size_t gsmem = row_smem_bytes(n, K);
    if (gsmem > (size_t)d->max_smem_optin) return DCP_ERR_UNSUPPORTED;
    const int grid = T < d->sms ? T : d->sms;
    // separate shards: scalar loads here, since this kernel does not check
    // the shards' alignment
    Source gsrc = src;
    if constexpr (Source::kIndirect) gsrc.vec4 = false;
    e = launch_serialized(topk_rows_kernel<Source>, grid, kThreads, gsmem, stream, gsrc, T, K,
                          out_scores, out_ids);
  }
  // the launch's own status only: an error left on the thread by unrelated
  // work is neither reported here nor cleared
  return e == cudaSuccess ? DCP_OK : DCP_ERR_CUDA;
}

}  // namespace dcp

extern "C" {

dcp_status dcp_topk_merge_workspace_size(int T, int dcp_, int K, size_t* bytes) {
  if (!bytes || T < 0 || dcp_ < 1 || K < 1) return DCP_ERR_INVALID;
  if (K > DCP_MAX_K || (long long)dcp_ * K > DCP_MAX_CANDIDATES) return DCP_ERR_UNSUPPORTED;
  *bytes = 0;
  return DCP_OK;
}

dcp_status dcp_topk_merge(const float* scores, const int32_t* ids, int T, int dcp_, int K,
                          const int32_t* row_starts, int32_t* out_ids, float* out_scores,
                          void* workspace, size_t workspace_bytes, dcp_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (T < 0 || dcp_ < 1 || K < 1) return DCP_ERR_INVALID;
  if (K > DCP_MAX_K || (long long)dcp_ * K > DCP_MAX_CANDIDATES) return DCP_ERR_UNSUPPORTED;
  if (T == 0) return DCP_OK;
  if (!scores || !ids || !out_ids || !out_scores) return DCP_ERR_INVALID;
  dcp::MergeSource src{scores, ids, nullptr, nullptr, row_starts, T, dcp_, K,
                       (K % 4) == 0 && dcp::aligned16(scores) && dcp::aligned16(ids)};
  return dcp::launch_rows(src, T, dcp_ * K, K, out_scores, out_ids, (cudaStream_t)stream);
}

// Whether `p` is memory the device can read (device, managed, or mapped
// host memory): a host-only pointer array would fault the kernel.
static bool device_readable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clears the error this query itself raised
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
         (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr);
}

dcp_status dcp_topk_merge_shards(const float* const* shard_scores, const int32_t* const* shard_ids,
                                 int T, int dcp_, int K, const int32_t* row_starts,
                                 int32_t* out_ids, float* out_scores, dcp_stream_t stream) {
  if (T < 0 || dcp_ < 1 || K < 1) return DCP_ERR_INVALID;
  if (K > DCP_MAX_K || (long long)dcp_ * K > DCP_MAX_CANDIDATES) return DCP_ERR_UNSUPPORTED;
  if (T == 0) return DCP_OK;
  if (!shard_scores || !shard_ids || !out_ids || !out_scores) return DCP_ERR_INVALID;
  if (!device_readable(shard_scores) || !device_readable(shard_ids)) return DCP_ERR_INVALID;
  // 16-byte paths when K allows them; the shard pointers themselves are
  // checked on the device (DCP_DEVICE_BAD_SHARD_ALIGNMENT)
  dcp::ShardsSource src{nullptr, nullptr, shard_scores, shard_ids, row_starts, T, dcp_, K,
                        (K % 4) == 0};
  return dcp::launch_rows(src, T, dcp_ * K, K, out_scores, out_ids, (cudaStream_t)stream);
}

dcp_status dcp_local_topk_ex(const float* logits, int T, int L, int ld, int K, int rank, int dcp_,
                             const int32_t* row_starts, int layout, float* out_scores,
                             int32_t* out_ids, dcp_stream_t stream) {
  if (T < 0 || L < 1 || ld < L || K < 1 || dcp_ < 1 || rank < 0 || rank >= dcp_ ||
      (layout != DCP_IDS_CONTIGUOUS && layout != DCP_IDS_INTERLEAVED))
    return DCP_ERR_INVALID;
  if (K > DCP_MAX_K || L > DCP_MAX_CANDIDATES) return DCP_ERR_UNSUPPORTED;
  if (T == 0) return DCP_OK;
  if (!logits || !out_scores || !out_ids) return DCP_ERR_INVALID;
  dcp::LocalSource src{};
  src.logits = logits;
  src.row_starts = row_starts;
  src.L = L;
  src.ld = ld;
  src.rank = rank;
  src.vec4 = (L % 4) == 0 && (ld % 4) == 0 && dcp::aligned16(logits);
  const bool inter = layout == DCP_IDS_INTERLEAVED;
  src.id_offset = inter ? (uint32_t)rank : (uint32_t)rank * (uint32_t)L;
  src.id_stride = inter ? (uint32_t)dcp_ : 1u;
  return dcp::launch_rows(src, T, L, K, out_scores, out_ids, (cudaStream_t)stream);
}

dcp_status dcp_local_topk(const float* logits, int T, int L, int ld, int K, int rank, int dcp_,
                          const int32_t* row_starts, float* out_scores, int32_t* out_ids,
                          dcp_stream_t stream) {
  return dcp_local_topk_ex(logits, T, L, ld, K, rank, dcp_, row_starts, DCP_IDS_CONTIGUOUS,
                           out_scores, out_ids, stream);
}

dcp_status dcp_fused_topk_ex(const float* logits, int T, int dcp_, int L, int ld, int K,
                             const int32_t* row_starts, int layout, float* out_scores,
                             int32_t* out_ids, dcp_stream_t stream) {
  if (T < 0 || dcp_ < 1 || L < 1 || ld < L || K < 1 ||
      (layout != DCP_IDS_CONTIGUOUS && layout != DCP_IDS_INTERLEAVED))
    return DCP_ERR_INVALID;
  if (K > DCP_MAX_K || (long long)dcp_ * L > DCP_MAX_CANDIDATES) return DCP_ERR_UNSUPPORTED;
  if (T == 0) return DCP_OK;
  if (!logits || !out_scores || !out_ids) return DCP_ERR_INVALID;
  dcp::FusedSource src{};
  src.logits = logits;
  src.row_starts = row_starts;
  src.T = T;
  src.dcp = dcp_;
  src.L = L;
  src.ld = ld;
  src.vec4 = (L % 4) == 0 && (ld % 4) == 0 && dcp::aligned16(logits);
  src.interleaved = layout == DCP_IDS_INTERLEAVED;
  src.l_recip = ((1ull << 32) + (unsigned long long)L - 1ull) / (unsigned long long)L;
  return dcp::launch_rows(src, T, dcp_ * L, K, out_scores, out_ids, (cudaStream_t)stream);
}

dcp_status dcp_fused_topk(const float* logits, int T, int dcp_, int L, int ld, int K,
                          const int32_t* row_starts, float* out_scores, int32_t* out_ids,
                          dcp_stream_t stream) {
  return dcp_fused_topk_ex(logits, T, dcp_, L, ld, K, row_starts, DCP_IDS_CONTIGUOUS, out_scores,
                           out_ids, stream);
}

dcp_status dcp_topk_device_status(unsigned int* status) {
  if (!status) return DCP_ERR_INVALID;
  unsigned int* word = nullptr;
  if (dcp::status_word(&word) != cudaSuccess) return DCP_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return DCP_ERR_CUDA;
  unsigned int v = 0u;
  if (cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DCP_ERR_CUDA;
  const unsigned int zero = 0u;
  if (cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return DCP_ERR_CUDA;
  *status = v;
  return DCP_OK;
}

dcp_status dcp_topk_selftest_wait_timeout(unsigned int wait_cycles, dcp_stream_t stream) {
  unsigned int* word = nullptr;
  if (dcp::status_word(&word) != cudaSuccess) return DCP_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1u);
  cfg.blockDim = dim3(32u);
  cfg.stream = (cudaStream_t)stream;
  const unsigned long long limit = wait_cycles;
  return cudaLaunchKernelEx(&cfg, dcp::wait_timeout_selftest_kernel, limit, word) == cudaSuccess
             ? DCP_OK
             : DCP_ERR_CUDA;
}

const char* dcp_status_string(dcp_status status) {
  switch (status) {
    case DCP_OK: return "DCP_OK";
    case DCP_ERR_INVALID: return "DCP_ERR_INVALID";
    case DCP_ERR_UNSUPPORTED: return "DCP_ERR_UNSUPPORTED";
    case DCP_ERR_CUDA: return "DCP_ERR_CUDA";
  }
  return "DCP_UNKNOWN_STATUS";
}

}  // extern "C"
