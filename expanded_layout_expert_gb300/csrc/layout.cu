// moe_expand_layout: per-expert histogram, aligned prefix, row labels and
// each pair's expanded row, computed on the device from topk_ids and the
// device-side valid-row count (SGLang PR 37261, "feat(deepep_v2): expanded
// (do_expand=True) prefill dispatch for DeepEP-V2": fill_m_indices_from_psum
// labels rows from the device psum with no cumsum, no H2D copy and no
// sentinel; the review thread fixes psum[i] = align(psum[i-1]) + count_i).
//
// Two launches, no spin-waits:
//  1. count: each block histograms a 2048-pair chunk into the workspace; the
//     last block to finish (atomic ticket, it never waits) scans the per-block
//     counts into per-(expert, block) base rows and the per-expert aligned
//     prefix, total and tile prefix.
//  2. rank: each block re-reads its chunk in (token, k) order, warp by warp,
//     and gives each valid pair base + rank (a stable counting sort); the
//     same blocks label m_indices by binary search over the segment starts.
// When every pair fits in one chunk (a decode-sized batch), one block does
// both passes in a single launch and no workspace is touched.
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPairsPerWarp = 256;
constexpr int kChunk = kWarps * kPairsPerWarp;  // pairs per block
constexpr int kMaxE = 1024;
constexpr int kPerThread = kChunk / kThreads;   // pairs per thread in the count pass
constexpr int kRounds = kPairsPerWarp / 32;     // 32-pair rounds per warp in the rank pass
constexpr int kScanSmem = 6144;                 // (expert, block) counts staged in shared memory

inline int64_t num_chunks(int64_t T, int K) {
  const int64_t pairs = T * K;
  const int64_t nb = (pairs + kChunk - 1) / kChunk;
  return nb > 0 ? nb : 1;
}

MOE_DEV int64_t valid_rows(const int32_t* d_n_valid, int64_t T) {
  if (d_n_valid == nullptr) return T;
  const int64_t nv = *d_n_valid;
  return nv < 0 ? 0 : (nv > T ? T : nv);
}

// Exclusive block-wide scan of one int per thread (kThreads threads).
MOE_DEV int block_exclusive_scan(int v, int* warp_tot, int* block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base += warp_tot[w];
    tot += warp_tot[w];
  }
  __syncthreads();
  *block_total = tot;
  return base + incl - v;
}

__global__ void __launch_bounds__(kThreads) layout_count_kernel(
    const int32_t* __restrict__ ids, int64_t T, int K, int E, int align,
    const int32_t* __restrict__ d_n_valid, int64_t M_cap, int nb, int32_t* __restrict__ counts,
    int32_t* __restrict__ offs, unsigned* __restrict__ ticket, int32_t* __restrict__ psum,
    int32_t* __restrict__ start, int32_t* __restrict__ d_total, int32_t* __restrict__ tile_prefix,
    int32_t* __restrict__ status) {
  __shared__ int hist[kMaxE];
  __shared__ int s_start[kMaxE];
  __shared__ int s_cnt[kScanSmem];
  __shared__ int warp_tot[kWarps];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();

  const int64_t npairs = valid_rows(d_n_valid, T) * K;
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kChunk;
  // all of this thread's ids first (independent loads), then the counting
  int idv[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int64_t p = p0 + j * kThreads + tid;
    idv[j] = (p < npairs) ? ids[p] : -1;
  }
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int id = idv[j];
    if (id >= E) set_status(status, MOE_ERR_DEVICE_CHECK);
    else if (id >= 0) atomicAdd(&hist[id], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) counts[static_cast<int64_t>(e) * nb + blockIdx.x] = hist[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(nb - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last block. The per-(expert, block) counts go through shared memory when
  // they fit (one round of parallel loads instead of a chain of dependent
  // ones); per expert, an exclusive scan over the blocks.
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t n_offs = static_cast<int64_t>(E) * nb;
  const bool staged = n_offs <= kScanSmem;
  if (staged) {
    for (int64_t i = tid; i < n_offs; i += kThreads) s_cnt[i] = __ldcg(&counts[i]);
    __syncthreads();
  }
  for (int e = warp; e < E; e += kWarps) {
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const int64_t i = static_cast<int64_t>(e) * nb + b;
      const int c = (b < nb) ? (staged ? s_cnt[i] : __ldcg(&counts[i])) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < nb) {
        if (staged) s_cnt[i] = carry + incl - c;
        else offs[i] = carry + incl - c;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) hist[e] = carry;  // count of expert e
  }
  __syncthreads();

  // Over experts: start[e] = sum_{j<e} align(count_j), psum[e] = start[e] +
  // count_e, tile prefix of ceil(align(count_e) / MOE_BLOCK_M).
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = tid * per;
  int rows_local = 0, tiles_local = 0;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      const int seg = align_up(hist[e], align);
      rows_local += seg;
      tiles_local += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
    }
  }
  int rows_total, tiles_total;
  int run = block_exclusive_scan(rows_local, warp_tot, &rows_total);
  int trun = block_exclusive_scan(tiles_local, warp_tot, &tiles_total);
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      const int c = hist[e];
      const int seg = align_up(c, align);
      start[e] = run;
      s_start[e] = run;
      psum[e] = run + c;
      tile_prefix[e] = trun;
      run += seg;
      trun += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
    }
  }
  if (tid == 0) {
    tile_prefix[E] = tiles_total;
    *d_total = rows_total;
    if (rows_total > M_cap) set_status(status, MOE_ERR_DEVICE_CHECK);
  }
  __syncthreads();
  if (staged) {
    for (int64_t i = tid; i < n_offs; i += kThreads) offs[i] = s_cnt[i] + s_start[i / nb];
  } else {
    for (int64_t i = tid; i < n_offs; i += kThreads) offs[i] += s_start[i / nb];
  }
  if (tid == 0) *ticket = 0u;  // ready for the next call
}

__global__ void __launch_bounds__(kThreads) layout_rank_kernel(
    const int32_t* __restrict__ ids, int64_t T, int K, int E, const int32_t* __restrict__ d_n_valid,
    int64_t M_cap, int nb, const int32_t* __restrict__ offs, const int32_t* __restrict__ start,
    const int32_t* __restrict__ d_total, int32_t* __restrict__ m_indices,
    int32_t* __restrict__ src2dst) {
  __shared__ int wcnt[kWarps * kMaxE];
  __shared__ int s_start[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  for (int e = tid; e < E; e += kThreads) s_start[e] = start[e];
  __syncthreads();

  const int64_t all_pairs = T * K;
  const int64_t npairs = valid_rows(d_n_valid, T) * K;
  const int64_t base_p = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kPairsPerWarp;
  int* my = wcnt + warp * E;

  // This warp's pairs, loaded up front (independent loads).
  int idv[kRounds];
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    idv[j] = (p < npairs) ? ids[p] : -1;
  }
  // Pass 1: this warp's pairs per expert.
#pragma unroll
  for (int j = 0; j < kRounds; ++j)
    if (idv[j] >= 0 && idv[j] < E) atomicAdd(&my[idv[j]], 1);
  __syncthreads();
  // Pass 2: per expert, exclusive over the warps, on top of the block's base.
  for (int e = tid; e < E; e += kThreads) {
    int acc = offs[static_cast<int64_t>(e) * nb + blockIdx.x];
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  // Pass 3: in (token, k) order, 32 pairs at a time; lanes holding the same
  // expert are ranked by lane, the lowest of them advances the counter.
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    const int id = idv[j];
    const bool valid = (id >= 0 && id < E);
    const int key = valid ? id : (E + static_cast<int>(lane));
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int dst = -1;
    if (valid) dst = my[id] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0u) my[id] += __popc(peers);
    __syncwarp();
    if (p < all_pairs) src2dst[p] = (dst >= 0 && dst < M_cap) ? dst : -1;
  }

  // Row labels: e on [start[e], start[e] + align(count_e)), -1 past the total.
  const int total = *d_total;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kThreads + tid; row < M_cap; row += stride) {
    int label = -1;
    if (row < total) {
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= row) lo = mid; else hi = mid - 1;
      }
      label = lo;
    }
    m_indices[row] = label;
  }
}

// Small inputs (all pairs in one 2048-pair chunk, e.g. a decode batch): the
// two passes above in one block and one launch. Count, scan over experts,
// stable ranks and row labels, with the per-(expert, warp) counters in
// dynamic shared memory (10 * E ints).
__global__ void __launch_bounds__(kThreads) layout_single_kernel(
    const int32_t* __restrict__ ids, int64_t T, int K, int E, int align,
    const int32_t* __restrict__ d_n_valid, int64_t M_cap, int32_t* __restrict__ psum,
    int32_t* __restrict__ start, int32_t* __restrict__ d_total, int32_t* __restrict__ tile_prefix,
    int32_t* __restrict__ m_indices, int32_t* __restrict__ src2dst, int32_t* __restrict__ status) {
  extern __shared__ int dyn[];
  int* hist = dyn;                 // [E] counts
  int* s_start = hist + E;         // [E]
  int* wcnt = s_start + E;         // [kWarps][E]
  __shared__ int warp_tot[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kThreads) hist[e] = 0;
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();

  const int64_t all_pairs = T * K;
  const int64_t npairs = valid_rows(d_n_valid, T) * K;
  // this warp's pairs in (token, k) order, loaded up front
  const int64_t base_p = static_cast<int64_t>(warp) * kPairsPerWarp;
  int idv[kRounds];
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    idv[j] = (p < npairs) ? ids[p] : -1;
  }
  int* my = wcnt + warp * E;
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int id = idv[j];
    if (id >= E) set_status(status, MOE_ERR_DEVICE_CHECK);
    else if (id >= 0) {
      atomicAdd(&hist[id], 1);
      atomicAdd(&my[id], 1);
    }
  }
  __syncthreads();

  // Over experts: start = sum of aligned counts before, psum = start + count,
  // the tile prefix and the total.
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = tid * per;
  int rows_local = 0, tiles_local = 0;
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      const int seg = align_up(hist[e], align);
      rows_local += seg;
      tiles_local += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
    }
  }
  int rows_total, tiles_total;
  int run = block_exclusive_scan(rows_local, warp_tot, &rows_total);
  int trun = block_exclusive_scan(tiles_local, warp_tot, &tiles_total);
  for (int j = 0; j < per; ++j) {
    const int e = e0 + j;
    if (e < E) {
      const int c = hist[e];
      const int seg = align_up(c, align);
      start[e] = run;
      s_start[e] = run;
      psum[e] = run + c;
      tile_prefix[e] = trun;
      run += seg;
      trun += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
    }
  }
  if (tid == 0) {
    tile_prefix[E] = tiles_total;
    *d_total = rows_total;
    if (rows_total > M_cap) set_status(status, MOE_ERR_DEVICE_CHECK);
  }
  __syncthreads();
  // per expert, each warp's first row: the segment start plus the earlier
  // warps' pairs of that expert
  for (int e = tid; e < E; e += kThreads) {
    int acc = s_start[e];
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  // stable ranks, 32 pairs at a time (lanes with the same expert ranked by lane)
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    const int id = idv[j];
    const bool valid = (id >= 0 && id < E);
    const int key = valid ? id : (E + static_cast<int>(lane));
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int dst = -1;
    if (valid) dst = my[id] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0u) my[id] += __popc(peers);
    __syncwarp();
    if (p < all_pairs) src2dst[p] = (dst >= 0 && dst < M_cap) ? dst : -1;
  }
  // row labels
  for (int64_t row = tid; row < M_cap; row += kThreads) {
    int label = -1;
    if (row < rows_total) {
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= row) lo = mid; else hi = mid - 1;
      }
      label = lo;
    }
    m_indices[row] = label;
  }
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_workspace_size(int64_t T, int K, int E) {
  if (T < 0 || K <= 0 || E <= 0) return 0;
  const int64_t nb = moe::num_chunks(T, K);
  const size_t tables = static_cast<size_t>(2) * static_cast<size_t>(E) * nb * sizeof(int32_t);
  return (tables + 255) / 256 * 256 + 256;  // + the ticket, in its own 256-byte slot
}

extern "C" int moe_expand_layout(const int32_t* topk_ids, int64_t T, int K, int E, int align,
                                 const int32_t* d_n_valid, int64_t M_cap, int32_t* psum,
                                 int32_t* start, int32_t* d_total, int32_t* m_indices,
                                 int32_t* src2dst, int32_t* tile_prefix, void* ws,
                                 size_t ws_bytes, int32_t* d_status, moe_stream_t stream) {
  MOE_REQUIRE(psum && start && d_total && tile_prefix, "moe_expand_layout: null output");
  MOE_REQUIRE(T == 0 || (topk_ids && src2dst), "moe_expand_layout: null topk_ids/src2dst");
  MOE_REQUIRE(M_cap == 0 || m_indices, "moe_expand_layout: null m_indices");
  MOE_REQUIRE(T >= 0 && K > 0 && E > 0 && E <= moe::kMaxE && align > 0 && M_cap >= 0,
              "moe_expand_layout: bad sizes T=%lld K=%d E=%d align=%d M_cap=%lld",
              (long long)T, K, E, align, (long long)M_cap);
  MOE_REQUIRE(T * K <= INT32_MAX && M_cap <= INT32_MAX, "moe_expand_layout: sizes exceed int32");
  MOE_REQUIRE_DEVICE();
  const size_t need = moe_workspace_size(T, K, E);
  if (ws == nullptr || ws_bytes < need) {
    moe::set_error("moe_expand_layout: workspace of %zu bytes needed", need);
    return MOE_ERR_WORKSPACE;
  }
  const int nb = static_cast<int>(moe::num_chunks(T, K));
  int32_t* counts = static_cast<int32_t*>(ws);
  int32_t* offs = counts + static_cast<int64_t>(E) * nb;
  unsigned* ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + need - 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nb == 1) {
    // every pair in one chunk: one block, one launch, no workspace
    const size_t smem = static_cast<size_t>(moe::kWarps + 2) * E * sizeof(int);
    moe::layout_single_kernel<<<1, moe::kThreads, smem, s>>>(topk_ids, T, K, E, align, d_n_valid,
                                                            M_cap, psum, start, d_total, tile_prefix,
                                                            m_indices, src2dst, d_status);
    return moe::check_launch("layout_single_kernel");
  }
  moe::layout_count_kernel<<<nb, moe::kThreads, 0, s>>>(topk_ids, T, K, E, align, d_n_valid, M_cap,
                                                        nb, counts, offs, ticket, psum, start,
                                                        d_total, tile_prefix, d_status);
  int rc = moe::check_launch("layout_count_kernel");
  if (rc != MOE_OK) return rc;
  moe::layout_rank_kernel<<<nb, moe::kThreads, 0, s>>>(topk_ids, T, K, E, d_n_valid, M_cap, nb,
                                                       offs, start, d_total, m_indices, src2dst);
  return moe::check_launch("layout_rank_kernel");
}

// ---------------------------------------------------------------------------
// moe_expand_layout_noalloc: the same two kernels, with their scratch in a
// fixed array that lives in the library's device image, so the caller passes
// no workspace and nothing is allocated on this path. Meant for callers that
// cannot allocate device memory at this point: a serving engine that has
// already handed all of HBM to its own pool, or a host loop that must not
// call cudaMalloc here because cudaMalloc can synchronise the device.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB per device

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device and CUDA
// context. In host code the array's name is only a host-side stand-in, never
// the device address, so kernels must be given this pointer instead. The
// cache is keyed on the current context as well as the device: after a
// device reset (or the primary context's teardown) the module is loaded
// again, the array may sit at another address, and the lookup is redone.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

struct NoAllocSlot {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
NoAllocSlot g_noalloc_slot[64];
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("moe_expand_layout_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) {
    set_error("moe_expand_layout_noalloc: device index %d out of range", dev);
    return MOE_ERR_UNSUPPORTED;
  }
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) {
    set_error("moe_expand_layout_noalloc: cuCtxGetCurrent is not available from the driver");
    return MOE_ERR_CUDA;
  }
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    set_error("moe_expand_layout_noalloc: no current CUDA context");
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc_slot[dev];
  if (slot.addr == nullptr || slot.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_error("moe_expand_layout_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    slot.ctx = ctx;
    slot.addr = p;
  }
  *out = slot.addr;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_expand_layout_noalloc_max_scratch(void) { return moe::kNoAllocScratchBytes; }

extern "C" int moe_expand_layout_noalloc(const int32_t* topk_ids, int64_t T, int K, int E,
                                         int align, const int32_t* d_n_valid, int64_t M_cap,
                                         int32_t* psum, int32_t* start, int32_t* d_total,
                                         int32_t* m_indices, int32_t* src2dst,
                                         int32_t* tile_prefix, int32_t* d_status,
                                         moe_stream_t stream) {
  MOE_REQUIRE(psum && start && d_total && tile_prefix, "moe_expand_layout_noalloc: null output");
  MOE_REQUIRE(T == 0 || (topk_ids && src2dst), "moe_expand_layout_noalloc: null topk_ids/src2dst");
  MOE_REQUIRE(M_cap == 0 || m_indices, "moe_expand_layout_noalloc: null m_indices");
  MOE_REQUIRE(T >= 0 && K > 0 && E > 0 && E <= moe::kMaxE && align > 0 && M_cap >= 0,
              "moe_expand_layout_noalloc: bad sizes T=%lld K=%d E=%d align=%d M_cap=%lld",
              (long long)T, K, E, align, (long long)M_cap);
  MOE_REQUIRE(T * K <= INT32_MAX && M_cap <= INT32_MAX,
              "moe_expand_layout_noalloc: sizes exceed int32");
  const size_t need = moe_workspace_size(T, K, E);
  MOE_REQUIRE(need <= moe::kNoAllocScratchBytes,
              "moe_expand_layout_noalloc: T=%lld K=%d E=%d needs %zu bytes of scratch, more than "
              "the fixed %zu; use moe_expand_layout with a workspace",
              (long long)T, K, E, need, moe::kNoAllocScratchBytes);
  MOE_REQUIRE_DEVICE();
  const int nb = static_cast<int>(moe::num_chunks(T, K));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nb == 1) {
    // every pair in one chunk: the one-launch layout, which needs no scratch
    const size_t smem = static_cast<size_t>(moe::kWarps + 2) * E * sizeof(int);
    moe::layout_single_kernel<<<1, moe::kThreads, smem, s>>>(topk_ids, T, K, E, align, d_n_valid,
                                                            M_cap, psum, start, d_total, tile_prefix,
                                                            m_indices, src2dst, d_status);
    return moe::check_launch("layout_single_kernel");
  }
  void* ws = nullptr;
  int rc = moe::noalloc_scratch(&ws);
  if (rc != MOE_OK) return rc;
  int32_t* counts = static_cast<int32_t*>(ws);
  int32_t* offs = counts + static_cast<int64_t>(E) * nb;
  unsigned* ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + need - 256);
  // The array keeps whatever the previous call left; the ticket must start
  // at zero (the counts and offsets are fully rewritten every call).
  cudaError_t e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) {
    moe::set_error("moe_expand_layout_noalloc: cudaMemsetAsync: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  moe::layout_count_kernel<<<nb, moe::kThreads, 0, s>>>(topk_ids, T, K, E, align, d_n_valid, M_cap,
                                                        nb, counts, offs, ticket, psum, start,
                                                        d_total, tile_prefix, d_status);
  rc = moe::check_launch("layout_count_kernel");
  if (rc != MOE_OK) return rc;
  moe::layout_rank_kernel<<<nb, moe::kThreads, 0, s>>>(topk_ids, T, K, E, d_n_valid, M_cap, nb,
                                                       offs, start, d_total, m_indices, src2dst);
  return moe::check_launch("layout_rank_kernel");
}

// ---------------------------------------------------------------------------
// moe_expand_layout_scatter: the layout fused into the scatter (SGLang PR
// 37261 names layout and scatter as the two light/heavy halves of the expand
// step; here they share launches). Launch 1 is layout_count_kernel above
// (per-chunk histograms, last-block scan). Launch 2 replaces both the rank
// pass and the stand-alone scatter: S blocks per 2048-pair chunk each rank
// the whole chunk exactly as layout_rank_kernel does (the ranks only need the
// chunk's base rows from launch 1, and redoing them costs a few KB of id
// reads), keep the destinations in shared memory and copy their share of the
// chunk's tokens: each token's fp8 row and scale row read once and stored to
// its destinations, with the pair's weight. The first of the S blocks writes
// src2dst; blocks placed first in the grid zero the alignment gaps; the chunk
// blocks label m_indices. The outputs are those of moe_expand_layout followed
// by moe_expand_scatter, bit for bit.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kPadRowsPerBlock = 8;

__global__ void __launch_bounds__(kThreads) layout_rank_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ topk_w,
    const uint4* __restrict__ x, const void* __restrict__ x_scale, int ue8m0, int64_t ld_xs,
    int64_t T, int H, int K, int E, int align, const int32_t* __restrict__ d_n_valid,
    int64_t M_cap, int nb, int S, const int32_t* __restrict__ offs,
    const int32_t* __restrict__ psum, const int32_t* __restrict__ start,
    const int32_t* __restrict__ d_total, int32_t* __restrict__ m_indices,
    int32_t* __restrict__ src2dst, uint4* __restrict__ xe, void* __restrict__ xe_scale,
    int64_t ld_xes, float* __restrict__ row_w, int pad_blocks_per_expert) {
  __shared__ int wcnt[kWarps * kMaxE];
  __shared__ int s_start[kMaxE];
  __shared__ int s_dst[kChunk];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nvec = H / 16;
  const int G = H / 128;
  const int W = (G + 3) / 4;
  const int pad_blocks = E * pad_blocks_per_expert;

  if (static_cast<int>(blockIdx.x) < pad_blocks) {
    // zero rows [psum[e], align(psum[e])) of expert e, 8 rows per block
    const int e = blockIdx.x / pad_blocks_per_expert;
    const int sub = blockIdx.x % pad_blocks_per_expert;
    const int64_t seg_end = align_up(psum[e], align);
    const int64_t r0 = static_cast<int64_t>(psum[e]) + static_cast<int64_t>(sub) * kPadRowsPerBlock;
    int64_t r1 = r0 + kPadRowsPerBlock;
    if (r1 > seg_end) r1 = seg_end;
    if (r1 > M_cap) r1 = M_cap;
    for (int64_t r = r0; r < r1; ++r) {
      for (int v = tid; v < nvec; v += kThreads) xe[r * nvec + v] = make_uint4(0, 0, 0, 0);
      if (!ue8m0) {
        for (int g = tid; g < G; g += kThreads) static_cast<float*>(xe_scale)[r * ld_xes + g] = 0.0f;
      } else {
        for (int j = tid; j < W; j += kThreads) static_cast<int32_t*>(xe_scale)[j * ld_xes + r] = 0;
      }
      if (tid == 0) row_w[r] = 0.0f;
    }
    return;
  }

  const int cb = blockIdx.x - pad_blocks;  // chunk block
  const int chunk = cb / S;
  const int part = cb % S;
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  for (int e = tid; e < E; e += kThreads) s_start[e] = start[e];
  __syncthreads();

  // --- ranks: the rank pass of layout_rank_kernel for this chunk
  const int64_t all_pairs = T * K;
  const int64_t npairs = valid_rows(d_n_valid, T) * K;
  const int64_t p0 = static_cast<int64_t>(chunk) * kChunk;
  const int64_t base_p = p0 + warp * kPairsPerWarp;
  int* my = wcnt + warp * E;
  int idv[kRounds];
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    idv[j] = (p < npairs) ? ids[p] : -1;
  }
#pragma unroll
  for (int j = 0; j < kRounds; ++j)
    if (idv[j] >= 0 && idv[j] < E) atomicAdd(&my[idv[j]], 1);
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    int acc = offs[static_cast<int64_t>(e) * nb + chunk];
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = acc;
      acc += c;
    }
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kRounds; ++j) {
    const int64_t p = base_p + j * 32 + lane;
    const int id = idv[j];
    const bool valid = (id >= 0 && id < E);
    const int key = valid ? id : (E + static_cast<int>(lane));
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int dst = -1;
    if (valid) dst = my[id] + __popc(peers & lt_mask);
    __syncwarp();
    if (valid && (peers & lt_mask) == 0u) my[id] += __popc(peers);
    __syncwarp();
    const int d = (dst >= 0 && dst < M_cap) ? dst : -1;
    s_dst[warp * kPairsPerWarp + j * 32 + lane] = d;
    if (part == 0 && p < all_pairs) src2dst[p] = d;
  }
  __syncthreads();

  // --- copy: tokens of this chunk's valid pairs, every S-th one from `part`
  int64_t p1 = p0 + kChunk;
  if (p1 > npairs) p1 = npairs;
  if (p1 > p0) {
    const int64_t t_first = p0 / K;
    const int64_t t_end = (p1 - 1) / K + 1;
    for (int64_t t = t_first + part; t < t_end; t += S) {
      const int64_t q0 = t * K;  // the token's first pair
      const int k_lo = q0 < p0 ? static_cast<int>(p0 - q0) : 0;
      const int k_hi = q0 + K > p1 ? static_cast<int>(p1 - q0) : K;
      const int kb0 = static_cast<int>(q0 - p0);  // s_dst[kb0 + k]: pair k of token t
      for (int v = tid; v < nvec; v += kThreads) {
        const uint4 val = __ldcs(x + t * nvec + v);
        for (int k = k_lo; k < k_hi; ++k) {
          const int r = s_dst[kb0 + k];
          if (r >= 0) xe[static_cast<int64_t>(r) * nvec + v] = val;
        }
      }
      if (!ue8m0) {
        const float* xs = static_cast<const float*>(x_scale);
        for (int g = tid; g < G; g += kThreads) {
          const float sv = xs[t * ld_xs + g];
          for (int k = k_lo; k < k_hi; ++k) {
            const int r = s_dst[kb0 + k];
            if (r >= 0) static_cast<float*>(xe_scale)[static_cast<int64_t>(r) * ld_xes + g] = sv;
          }
        }
      } else {
        const int32_t* xs = static_cast<const int32_t*>(x_scale);
        for (int j = tid; j < W; j += kThreads) {
          const int32_t wv = xs[j * ld_xs + t];
          for (int k = k_lo; k < k_hi; ++k) {
            const int r = s_dst[kb0 + k];
            if (r >= 0) static_cast<int32_t*>(xe_scale)[j * ld_xes + r] = wv;
          }
        }
      }
      if (tid >= k_lo && tid < k_hi && s_dst[kb0 + tid] >= 0) row_w[s_dst[kb0 + tid]] = topk_w[q0 + tid];
    }
  }

  // --- row labels: e on [start[e], start[e] + align(count_e)), -1 past the total
  const int total = *d_total;
  const int64_t nchunk_blocks = static_cast<int64_t>(gridDim.x) - pad_blocks;
  for (int64_t row = static_cast<int64_t>(cb) * kThreads + tid; row < M_cap;
       row += nchunk_blocks * kThreads) {
    int label = -1;
    if (row < total) {
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= row) lo = mid; else hi = mid - 1;
      }
      label = lo;
    }
    m_indices[row] = label;
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_expand_layout_scatter(
    const int32_t* topk_ids, const float* topk_w, const uint8_t* x, const void* x_scale,
    int scale_layout, int64_t ld_xs, int64_t T, int H, int K, int E, int align,
    const int32_t* d_n_valid, int64_t M_cap, int32_t* psum, int32_t* start, int32_t* d_total,
    int32_t* m_indices, int32_t* src2dst, int32_t* tile_prefix, uint8_t* xe, void* xe_scale,
    int64_t ld_xes, float* row_w, void* ws, size_t ws_bytes, int32_t* d_status,
    moe_stream_t stream) {
  MOE_REQUIRE(psum && start && d_total && tile_prefix && xe && xe_scale && row_w,
              "moe_expand_layout_scatter: null output");
  MOE_REQUIRE(T == 0 || (topk_ids && topk_w && x && x_scale && src2dst),
              "moe_expand_layout_scatter: null input");
  MOE_REQUIRE(M_cap == 0 || m_indices, "moe_expand_layout_scatter: null m_indices");
  MOE_REQUIRE(T >= 0 && K > 0 && K <= 32 && E > 0 && E <= moe::kMaxE && align > 0 && M_cap >= 0,
              "moe_expand_layout_scatter: bad sizes T=%lld K=%d E=%d align=%d M_cap=%lld",
              (long long)T, K, E, align, (long long)M_cap);
  MOE_REQUIRE(T * K <= INT32_MAX && M_cap <= INT32_MAX,
              "moe_expand_layout_scatter: sizes exceed int32");
  MOE_REQUIRE(H > 0 && H % 128 == 0 && H <= 16384,
              "moe_expand_layout_scatter: H must be a multiple of 128, <= 16384");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_expand_layout_scatter: bad scale layout");
  const int G = H / 128;
  if (scale_layout == MOE_SCALE_F32_ROWMAJOR) {
    MOE_REQUIRE(ld_xs >= G && ld_xes >= G,
                "moe_expand_layout_scatter: scale leading dimension < H/128");
  } else {
    MOE_REQUIRE(ld_xs >= T && ld_xes >= M_cap,
                "moe_expand_layout_scatter: packed scale leading dimension < rows");
  }
  MOE_REQUIRE(moe::aligned(x, 16) && moe::aligned(xe, 16),
              "moe_expand_layout_scatter: x/xe not 16-byte aligned");
  MOE_REQUIRE_DEVICE();
  const size_t need = moe_workspace_size(T, K, E);
  if (ws == nullptr || ws_bytes < need) {
    moe::set_error("moe_expand_layout_scatter: workspace of %zu bytes needed", need);
    return MOE_ERR_WORKSPACE;
  }
  const int nb = static_cast<int>(moe::num_chunks(T, K));
  int32_t* counts = static_cast<int32_t*>(ws);
  int32_t* offs = counts + static_cast<int64_t>(E) * nb;
  unsigned* ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + need - 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  moe::layout_count_kernel<<<nb, moe::kThreads, 0, s>>>(topk_ids, T, K, E, align, d_n_valid, M_cap,
                                                        nb, counts, offs, ticket, psum, start,
                                                        d_total, tile_prefix, d_status);
  int rc = moe::check_launch("layout_count_kernel");
  if (rc != MOE_OK) return rc;
  // S blocks per chunk: about four blocks per SM in all, and no more blocks
  // per chunk than the chunk has tokens
  int64_t tokens_per_chunk = (moe::kChunk + K - 1) / K + 1;
  if (tokens_per_chunk > T + 1) tokens_per_chunk = T + 1;
  int S = (4 * moe::device_sm_count() + nb - 1) / nb;
  if (S > tokens_per_chunk) S = static_cast<int>(tokens_per_chunk);
  if (S < 1) S = 1;
  const int pad_per_expert = (align - 1 + moe::kPadRowsPerBlock - 1) / moe::kPadRowsPerBlock;
  const int64_t grid = static_cast<int64_t>(E) * pad_per_expert + static_cast<int64_t>(nb) * S;
  MOE_REQUIRE(grid < (1ll << 31), "moe_expand_layout_scatter: grid too large");
  moe::layout_rank_scatter_kernel<<<static_cast<unsigned>(grid), moe::kThreads, 0, s>>>(
      topk_ids, topk_w, reinterpret_cast<const uint4*>(x), x_scale,
      scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR, ld_xs, T, H, K, E, align, d_n_valid, M_cap,
      nb, S, offs, psum, start, d_total, m_indices, src2dst, reinterpret_cast<uint4*>(xe), xe_scale,
      ld_xes, row_w, pad_per_expert);
  return moe::check_launch("layout_rank_scatter_kernel");
}
