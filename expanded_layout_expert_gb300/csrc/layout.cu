// moe_expand_layout: per-expert histogram, aligned prefix, row labels and
// each pair's expanded row, computed on the device from topk_ids and the
// device-side valid-row count (SGLang PR 37261, "feat(deepep_v2): expanded
// (do_expand=True) prefill dispatch for DeepEP-V2": fill_m_indices_from_psum
// labels rows from the device psum with no cumsum, no H2D copy and no
// sentinel; the review thread fixes psum[i] = align(psum[i-1]) + count_i).
//
// Three forms, the same outputs bit for bit, all a stable counting sort of
// the pairs in (token, k) order over 2048-pair chunks:
//  - one chunk (a decode-sized batch): one block, one launch, no workspace;
//  - several chunks that a cooperative grid holds: one launch of one block
//    per chunk with a bounded grid-wide barrier between counting and
//    ranking (layout_coop_kernel, below; fused with the expand-scatter it
//    is also the scatter's launch);
//  - more chunks: two launches without any wait.
//     1. count: each block histograms its chunk into the workspace; the last
//        block to finish (atomic ticket, it never waits) scans the per-block
//        counts into per-(expert, block) base rows and the per-expert
//        aligned prefix, total and tile prefix.
//     2. rank: each block re-reads its chunk in (token, k) order, warp by
//        warp, and gives each valid pair base + rank; the same blocks label
//        m_indices by binary search over the segment starts.
#include <atomic>
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

// ---------------------------------------------------------------------------
// The layout (and the layout fused with the expand-scatter) in ONE launch.
// A cooperative launch puts every block on the GPU at once, so blocks may
// wait for each other at a grid-wide barrier (bounded, like every wait in
// this library). Blocks 0 .. nb-1 own one 2048-pair chunk each (16 warps):
//   A. each warp ranks its 128 pairs among themselves (match_any groups
//      the lanes holding one expert; the lowest lane advances the warp's
//      counter), then the block turns the per-warp counts into per-warp
//      offsets and publishes the chunk's count per expert;
//   -- barrier of the chunk blocks --
//   C. every chunk block reads the whole count table (E x chunks, from L2,
//      a group of lanes per expert) and derives the expert totals, the
//      aligned segment starts (one block-wide scan over the experts) and
//      its own chunk's first row per expert;
//   D. it writes src2dst of its chunk: segment start + earlier chunks +
//      earlier warps + the rank inside the warp;
//   E. the chunk blocks label m_indices, four consecutive rows per thread
//      and one search per four rows.
// Fused with the scatter, the grid has more blocks than chunks; the others
// go straight to the second barrier, which all blocks meet:
//   -- barrier of all blocks --
//   F. the whole grid zeroes the alignment gaps, then copies every valid
//      token's row, scale row and weight to its expanded rows. The copy's
//      work items are 1 KB pieces of a token's row; warps take them from a
//      shared counter, kCopyGrab at a time, so the grid finishes together.
// The outputs equal those of the two-launch layout (and of
// moe_expand_scatter) bit for bit. The four barrier and counter words live
// in the workspace's ticket slot; the last block to leave resets them.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int kCoopThreads = 512;
constexpr int kCoopWarps = kCoopThreads / 32;
constexpr int kCoopPairsPerWarp = kChunk / kCoopWarps;  // 128
constexpr int kCoopRounds = kCoopPairsPerWarp / 32;     // 4
constexpr int kCoopMaxK = 32;
constexpr int kCoopPadRows = 8;        // gap rows per work item of the copy phase
constexpr int kCopyU = 2;              // 16-byte vectors per lane in flight in the copy
constexpr int kCopyPiece = 32 * kCopyU;  // vectors per work item of the copy
constexpr int kCopyGrab = 4;           // work items a warp takes per counter update
// Words of the 256-byte ticket slot: barrier 1 (also the two-launch path's
// ticket) and the exit count share the first 128-byte line; barrier 2 and
// the copy's work counter are in the second, so blocks polling barrier 2
// do not slow the traffic on barrier 1.
constexpr int kBar1Word = 0, kExitWord = 8, kBar2Word = 32, kWorkWord = 48;
constexpr size_t kSyncSlotBytes = 256;

MOE_DEV unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch: every block arrives once
// (after its writes, released to the GPU), thread 0 waits until `target`
// arrivals in all, sleeping sleep_ns between polls. Gives up after
// kWaitLimitCycles with MOE_ERR_TIMEOUT; returns false then.
MOE_DEV bool grid_sync(unsigned* arrivals, unsigned target, int32_t* status, int* s_flag,
                       unsigned sleep_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" : : "l"(arrivals) : "memory");
    int ok = 1;
    const long long t0 = clock64();
    while (ld_acquire_u32(arrivals) < target) {
      if (sleep_ns) __nanosleep(sleep_ns);
      if (clock64() - t0 > kWaitLimitCycles) {
        set_status(status, MOE_ERR_TIMEOUT);
        ok = 0;
        break;
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Exclusive scan of two ints per thread over the kCoopThreads threads:
// {prefix of a, prefix of b, total of a, total of b}.
MOE_DEV int4 coop_exclusive_scan2(int a, int b, int2* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, ia, o);
    const int yb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ya;
      ib += yb;
    }
  }
  if (lane == 31) warp_tot[warp] = make_int2(ia, ib);
  __syncthreads();
  int ba = 0, bb = 0, ta = 0, tb = 0;
#pragma unroll
  for (int w = 0; w < kCoopWarps; ++w) {
    const int2 v = warp_tot[w];
    if (w < warp) {
      ba += v.x;
      bb += v.y;
    }
    ta += v.x;
    tb += v.y;
  }
  __syncthreads();
  return make_int4(ba + ia - a, bb + ib - b, ta, tb);
}

// m_indices rows [r, r + 4) for r = first, first + stride, ...: e on
// [start[e], start[e] + align(count_e)), -1 past the total; one search per
// four rows.
MOE_DEV void label_rows(int32_t* m_indices, int64_t M_cap, int total, const int* s_start, int E,
                        int64_t first, int64_t stride) {
  for (int64_t r0 = first; r0 < M_cap; r0 += stride) {
    int e = 0;
    if (r0 < total) {
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= r0) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + i;
      if (row >= M_cap) break;
      if (row < total) {
        while (e + 1 < E && s_start[e + 1] <= row) ++e;
        m_indices[row] = e;
      } else {
        m_indices[row] = -1;
      }
    }
  }
}

struct CoopScatterArgs {
  const float* topk_w;
  const uint4* x;
  const void* x_scale;
  int ue8m0;
  int64_t ld_xs;
  int H;
  uint4* xe;
  void* xe_scale;
  int64_t ld_xes;
  float* row_w;
};

template <bool kScatter>
__global__ void __launch_bounds__(kCoopThreads, kScatter ? 2 : 3) layout_coop_kernel(
    const int32_t* __restrict__ ids, int64_t T, int K, int E, int align,
    const int32_t* __restrict__ d_n_valid, int64_t M_cap, int nb, int32_t* __restrict__ counts,
    unsigned* __restrict__ sync_words, int32_t* __restrict__ psum, int32_t* __restrict__ start,
    int32_t* __restrict__ d_total, int32_t* __restrict__ tile_prefix,
    int32_t* __restrict__ m_indices, int32_t* __restrict__ src2dst, int32_t* __restrict__ status,
    const CoopScatterArgs sa) {
  extern __shared__ int dyn[];
  int* hist = dyn;                 // [E] expert totals
  int* s_start = hist + E;         // [E] segment starts
  int* s_base = s_start + E;       // [E] this chunk's first row per expert
  int* wcnt = s_base + E;          // [kCoopWarps][E] per-warp counts, then offsets
  __shared__ int2 warp_tot[kCoopWarps];
  __shared__ int s_flag, s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = static_cast<int>(blockIdx.x);
  const int64_t nv = valid_rows(d_n_valid, T);
  unsigned* bar1 = sync_words + kBar1Word;
  unsigned* exits = sync_words + kExitWord;
  bool ok = true;

  if (b < nb) {  // block-uniform: a chunk block
    const int64_t all_pairs = T * K;
    const int64_t npairs = nv * K;
    const unsigned lt_mask = (1u << lane) - 1u;

    // A: ranks inside each warp, per-warp offsets, the chunk's counts
    for (int i = tid; i < kCoopWarps * E; i += kCoopThreads) wcnt[i] = 0;
    __syncthreads();
    const int64_t base_p = static_cast<int64_t>(b) * kChunk + warp * kCoopPairsPerWarp;
    // per pair: expert << 8 | rank inside the warp (< 128), or -1
    int rk[kCoopRounds];
#pragma unroll
    for (int j = 0; j < kCoopRounds; ++j) {
      const int64_t p = base_p + j * 32 + lane;
      rk[j] = p < npairs ? ids[p] : -1;
    }
    int* my = wcnt + warp * E;
#pragma unroll
    for (int j = 0; j < kCoopRounds; ++j) {
      const int id = rk[j];
      if (id >= E) set_status(status, MOE_ERR_DEVICE_CHECK);
      const bool valid = (id >= 0 && id < E);
      const int key = valid ? id : (E + static_cast<int>(lane));
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      rk[j] = valid ? (id << 8) | (my[id] + __popc(peers & lt_mask)) : -1;
      __syncwarp();
      if (valid && (peers & lt_mask) == 0u) my[id] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < E; e += kCoopThreads) {
      int acc = 0;
#pragma unroll
      for (int w = 0; w < kCoopWarps; ++w) {
        const int c = wcnt[w * E + e];
        wcnt[w * E + e] = acc;
        acc += c;
      }
      counts[static_cast<int64_t>(e) * nb + b] = acc;
    }

    ok = grid_sync(bar1, nb, status, &s_flag, 0);
    if (ok) {
      // C: per expert the total and the count of the chunks before this
      // one; gsz lanes (a power of two) share an expert
      int gsz = 32;
      while (gsz > 1 && gsz * E > kCoopThreads) gsz >>= 1;
      const int ngroups = kCoopThreads / gsz;
      const int gl = tid & (gsz - 1);
      for (int e0 = 0; e0 < E; e0 += ngroups) {  // uniform trip count
        const int e = e0 + tid / gsz;
        int tot = 0, pre = 0;
        if (e < E) {
          const int32_t* row = counts + static_cast<int64_t>(e) * nb;
          for (int c = gl; c < nb; c += 4 * gsz) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int cc = c + u * gsz;
              v[u] = cc < nb ? __ldcg(row + cc) : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              tot += v[u];
              if (c + u * gsz < b) pre += v[u];
            }
          }
        }
        for (int o = gsz >> 1; o > 0; o >>= 1) {
          tot += __shfl_xor_sync(0xffffffffu, tot, o);
          pre += __shfl_xor_sync(0xffffffffu, pre, o);
        }
        if (e < E && gl == 0) {
          hist[e] = tot;
          s_base[e] = pre;
        }
      }
      __syncthreads();
      // segment starts and tile prefix: one scan over the experts of
      // (aligned rows, tiles), every thread a contiguous run of experts
      {
        const int per = (E + kCoopThreads - 1) / kCoopThreads;
        const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
        int rows = 0, tiles = 0;
        for (int e = e_lo; e < e_hi; ++e) {
          const int seg = align_up(hist[e], align);
          rows += seg;
          tiles += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
        }
        const int4 sc = coop_exclusive_scan2(rows, tiles, warp_tot);
        int run = sc.x, trun = sc.y;
        for (int e = e_lo; e < e_hi; ++e) {
          const int c = hist[e];
          const int seg = align_up(c, align);
          s_start[e] = run;
          s_base[e] += run;
          if (b == 0) {
            start[e] = run;
            psum[e] = run + c;
            tile_prefix[e] = trun;
          }
          run += seg;
          trun += (seg + MOE_BLOCK_M - 1) / MOE_BLOCK_M;
        }
        if (tid == 0) {
          s_total = sc.z;
          if (b == 0) {
            tile_prefix[E] = sc.w;
            *d_total = sc.z;
            if (sc.z > M_cap) set_status(status, MOE_ERR_DEVICE_CHECK);
          }
        }
      }
      __syncthreads();

      // D: src2dst of this chunk's pairs
#pragma unroll
      for (int j = 0; j < kCoopRounds; ++j) {
        const int64_t p = base_p + j * 32 + lane;
        int dst = -1;
        if (rk[j] >= 0) {
          const int id = rk[j] >> 8;
          dst = s_base[id] + my[id] + (rk[j] & 0xff);
        }
        if (p < all_pairs) src2dst[p] = (dst >= 0 && dst < M_cap) ? dst : -1;
      }

      // E: row labels (the fused kernel labels them after its second
      // barrier, with the whole grid)
      if (!kScatter)
        label_rows(m_indices, M_cap, s_total, s_start, E,
                   (static_cast<int64_t>(b) * kCoopThreads + tid) * 4,
                   static_cast<int64_t>(nb) * kCoopThreads * 4);
    }
  }

  if constexpr (kScatter) {
    unsigned* bar2 = sync_words + kBar2Word;
    unsigned* work = sync_words + kWorkWord;
    if (ok) ok = grid_sync(bar2, gridDim.x, status, &s_flag, 128);
    if (ok) {
      // E: row labels from the published segment starts
      for (int e = tid; e < E; e += kCoopThreads) s_start[e] = __ldcg(&start[e]);
      if (tid == 0) s_total = __ldcg(d_total);
      __syncthreads();
      label_rows(m_indices, M_cap, s_total, s_start, E,
                 (static_cast<int64_t>(b) * kCoopThreads + tid) * 4,
                 static_cast<int64_t>(gridDim.x) * kCoopThreads * 4);
      const int H = sa.H;
      const int nvec = H / 16;
      const int G = H / 128;
      const int W = (G + 3) / 4;
      // F1: alignment gaps [psum[e], align(psum[e])), 8 rows per work item
      const int per_e = (align - 1 + kCoopPadRows - 1) / kCoopPadRows;
      const int items = E * per_e;
      for (int it = b; it < items; it += gridDim.x) {
        const int e = it / per_e, sub = it % per_e;
        const int pe = __ldcg(&psum[e]);
        const int64_t seg_end = align_up(pe, align);
        const int64_t r0 = static_cast<int64_t>(pe) + static_cast<int64_t>(sub) * kCoopPadRows;
        int64_t r1 = r0 + kCoopPadRows;
        if (r1 > seg_end) r1 = seg_end;
        if (r1 > M_cap) r1 = M_cap;
        for (int64_t r = r0; r < r1; ++r) {
          for (int v = tid; v < nvec; v += kCoopThreads) sa.xe[r * nvec + v] = make_uint4(0, 0, 0, 0);
          if (!sa.ue8m0) {
            for (int g = tid; g < G; g += kCoopThreads)
              static_cast<float*>(sa.xe_scale)[r * sa.ld_xes + g] = 0.0f;
          } else {
            for (int j = tid; j < W; j += kCoopThreads)
              static_cast<int32_t*>(sa.xe_scale)[j * sa.ld_xes + r] = 0;
          }
          if (tid == 0) sa.row_w[r] = 0.0f;
        }
      }
      // F2: work items (token, piece of kCopyPiece vectors) from the shared
      // counter. Lane k < K holds pair k's row; every lane loads kCopyU
      // vectors of the piece before storing them to the K rows. The first
      // piece of a token also copies its scales and weights.
      const int nseg = (nvec + kCopyPiece - 1) / kCopyPiece;
      const int64_t n_items = nv * nseg;
      for (;;) {
        unsigned grab = 0;  // the host keeps the counter's range inside 32 bits
        if (lane == 0) grab = atomicAdd(work, static_cast<unsigned>(kCopyGrab));
        grab = __shfl_sync(0xffffffffu, grab, 0);
        if (static_cast<int64_t>(grab) >= n_items) break;
        const int64_t it_end = min(n_items, static_cast<int64_t>(grab) + kCopyGrab);
        for (int64_t it = static_cast<int64_t>(grab); it < it_end; ++it) {
          const int64_t t = it / nseg;
          const int v0 = static_cast<int>(it - t * nseg) * kCopyPiece;
          int r = -1;
          if (lane < K) {
            r = __ldcg(&src2dst[t * K + lane]);
            if (r >= M_cap) {
              set_status(status, MOE_ERR_DEVICE_CHECK);
              r = -1;
            }
          }
          const uint4* src = sa.x + t * nvec;
          uint4 val[kCopyU];
#pragma unroll
          for (int u = 0; u < kCopyU; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) val[u] = __ldcs(src + v);
          }
          for (int k = 0; k < K; ++k) {
            const int rk = __shfl_sync(0xffffffffu, r, k);
            if (rk < 0) continue;
            uint4* dst = sa.xe + static_cast<int64_t>(rk) * nvec;
#pragma unroll
            for (int u = 0; u < kCopyU; ++u) {
              const int v = v0 + u * 32 + lane;
              if (v < nvec) dst[v] = val[u];
            }
          }
          if (v0 != 0) continue;
          if (!sa.ue8m0) {
            const float* xs = static_cast<const float*>(sa.x_scale);
            float* ys = static_cast<float*>(sa.xe_scale);
            for (int c0 = 0; c0 < G; c0 += 32) {
              const int c = c0 + lane;
              const float sv = c < G ? xs[t * sa.ld_xs + c] : 0.0f;
              for (int k = 0; k < K; ++k) {
                const int rk = __shfl_sync(0xffffffffu, r, k);
                if (rk >= 0 && c < G) ys[static_cast<int64_t>(rk) * sa.ld_xes + c] = sv;
              }
            }
          } else {
            const int32_t* xs = static_cast<const int32_t*>(sa.x_scale);
            int32_t* ys = static_cast<int32_t*>(sa.xe_scale);
            for (int j0 = 0; j0 < W; j0 += 32) {
              const int j = j0 + lane;
              const int32_t wv = j < W ? xs[j * sa.ld_xs + t] : 0;
              for (int k = 0; k < K; ++k) {
                const int rk = __shfl_sync(0xffffffffu, r, k);
                if (rk >= 0 && j < W) ys[j * sa.ld_xes + rk] = wv;
              }
            }
          }
          if (r >= 0) sa.row_w[r] = sa.topk_w[t * K + lane];
        }
      }
    }
  }

  // the last block to leave makes the barrier and counter words ready for
  // the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(exits, 1u) == gridDim.x - 1) {
      atomicExch(bar1, 0u);
      atomicExch(exits, 0u);
      atomicExch(sync_words + kBar2Word, 0u);
      atomicExch(sync_words + kWorkWord, 0u);
    }
  }
}

size_t coop_smem_bytes(int E) {
  return static_cast<size_t>(3 * E + kCoopWarps * E) * sizeof(int);
}

// Largest grid a cooperative launch of the kernel can have (all blocks
// resident), or 0 if the query fails. The answer for the last shared-memory
// size asked is kept per device (the layer asks the same size every call)
// when that size needs no function attribute (<= 48 KB, E <= 646), which a
// new context would have lost.
template <bool kScatter>
int coop_capacity(size_t smem) {
  constexpr int kDevices = 64;
  static std::atomic<int64_t> cached[kDevices];  // smem << 32 | capacity, 0 = none
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const bool cacheable = dev >= 0 && dev < kDevices && smem <= 48 * 1024;
  if (cacheable) {
    const int64_t c = cached[dev].load(std::memory_order_relaxed);
    if (c != 0 && static_cast<size_t>(c >> 32) == smem) return static_cast<int>(c & 0xFFFFFFFF);
  }
  auto kernel = layout_coop_kernel<kScatter>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCoopThreads, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int cap = per_sm * device_sm_count();
  if (cacheable && cap > 0)
    cached[dev].store((static_cast<int64_t>(smem) << 32) | cap, std::memory_order_relaxed);
  return cap;
}

template <bool kScatter>
int launch_coop(int grid, size_t smem, cudaStream_t s, const int32_t* ids, int64_t T, int K,
                int E, int align, const int32_t* d_n_valid, int64_t M_cap, int nb,
                int32_t* counts, unsigned* sync_words, int32_t* psum, int32_t* start,
                int32_t* d_total, int32_t* tile_prefix, int32_t* m_indices, int32_t* src2dst,
                int32_t* status, const CoopScatterArgs& sa) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, layout_coop_kernel<kScatter>, ids, T, K, E, align,
                                           d_n_valid, M_cap, nb, counts, sync_words, psum, start,
                                           d_total, tile_prefix, m_indices, src2dst, status, sa);
  if (e != cudaSuccess) {
    set_error("layout_coop_kernel: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return check_launch("layout_coop_kernel");
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// The layout of more than one chunk: one cooperative launch when the count
// matrix fits in shared memory and every chunk's block can be resident at
// once, else the count/scan launch and the rank launch. Both give the same
// outputs bit for bit. sync_words: the zeroed 256-byte ticket slot.
int layout_multi_chunk(const int32_t* ids, int64_t T, int K, int E, int align,
                       const int32_t* d_n_valid, int64_t M_cap, int nb, int32_t* counts,
                       int32_t* offs, unsigned* ticket, int32_t* psum, int32_t* start,
                       int32_t* d_total, int32_t* tile_prefix, int32_t* m_indices,
                       int32_t* src2dst, int32_t* d_status, cudaStream_t s) {
  const size_t smem = coop_smem_bytes(E);
  if (coop_capacity<false>(smem) >= nb) {
    const CoopScatterArgs none = {};
    return launch_coop<false>(nb, smem, s, ids, T, K, E, align, d_n_valid, M_cap, nb, counts,
                              ticket, psum, start, d_total, tile_prefix, m_indices, src2dst,
                              d_status, none);
  }
  layout_count_kernel<<<nb, kThreads, 0, s>>>(ids, T, K, E, align, d_n_valid, M_cap, nb, counts,
                                              offs, ticket, psum, start, d_total, tile_prefix,
                                              d_status);
  int rc = check_launch("layout_count_kernel");
  if (rc != MOE_OK) return rc;
  layout_rank_kernel<<<nb, kThreads, 0, s>>>(ids, T, K, E, d_n_valid, M_cap, nb, offs, start,
                                             d_total, m_indices, src2dst);
  return check_launch("layout_rank_kernel");
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_workspace_size(int64_t T, int K, int E) {
  if (T < 0 || K <= 0 || E <= 0) return 0;
  const int64_t nb = moe::num_chunks(T, K);
  const size_t tables = static_cast<size_t>(2) * static_cast<size_t>(E) * nb * sizeof(int32_t);
  return 256 + (tables + 255) / 256 * 256;  // the ticket slot, then the tables
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
  unsigned* ticket = static_cast<unsigned*>(ws);  // the first 256 bytes, whatever T is
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
  int32_t* offs = counts + static_cast<int64_t>(E) * nb;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (nb == 1) {
    // every pair in one chunk: one block, one launch, no workspace
    const size_t smem = static_cast<size_t>(moe::kWarps + 2) * E * sizeof(int);
    moe::layout_single_kernel<<<1, moe::kThreads, smem, s>>>(topk_ids, T, K, E, align, d_n_valid,
                                                            M_cap, psum, start, d_total, tile_prefix,
                                                            m_indices, src2dst, d_status);
    return moe::check_launch("layout_single_kernel");
  }
  return moe::layout_multi_chunk(topk_ids, T, K, E, align, d_n_valid, M_cap, nb, counts, offs,
                                 ticket, psum, start, d_total, tile_prefix, m_indices, src2dst,
                                 d_status, s);
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
  unsigned* ticket = static_cast<unsigned*>(ws);  // the first 256 bytes, whatever T is
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
  int32_t* offs = counts + static_cast<int64_t>(E) * nb;
  // The array keeps whatever the previous call left; the ticket and the
  // barrier words beside it must start at zero (the counts and offsets are
  // fully rewritten every call).
  cudaError_t e = cudaMemsetAsync(ticket, 0, moe::kSyncSlotBytes, s);
  if (e != cudaSuccess) {
    moe::set_error("moe_expand_layout_noalloc: cudaMemsetAsync: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return moe::layout_multi_chunk(topk_ids, T, K, E, align, d_n_valid, M_cap, nb, counts, offs,
                                 ticket, psum, start, d_total, tile_prefix, m_indices, src2dst,
                                 d_status, s);
}

// ---------------------------------------------------------------------------
// moe_expand_layout_scatter: the layout fused into the scatter (SGLang PR
// 37261 names layout and scatter as the two light/heavy halves of the expand
// step). When the cooperative grid holds every chunk: layout_coop_kernel
// <true>, one launch. Otherwise (one chunk, or more chunks than the grid
// holds) moe_expand_layout followed by moe_expand_scatter. The outputs are
// the same bit for bit either way.
// ---------------------------------------------------------------------------
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
  unsigned* ticket = static_cast<unsigned*>(ws);  // the first 256 bytes, whatever T is
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto layout_then_scatter = [&]() {
    const int rc = moe_expand_layout(topk_ids, T, K, E, align, d_n_valid, M_cap, psum, start,
                                     d_total, m_indices, src2dst, tile_prefix, ws, ws_bytes,
                                     d_status, stream);
    if (rc != MOE_OK) return rc;
    return moe_expand_scatter(x, x_scale, scale_layout, ld_xs, topk_w, src2dst, psum, start,
                              d_n_valid, T, H, K, E, align, M_cap, xe, xe_scale, ld_xes, row_w,
                              d_status, stream);
  };
  // every pair in one chunk: the one-block layout, then the scatter
  if (nb == 1) return layout_then_scatter();
  if (K <= moe::kCoopMaxK) {
    // one cooperative launch: layout, grid barrier, copy with the whole grid
    const size_t smem = moe::coop_smem_bytes(E);
    const int cap = moe::coop_capacity<true>(smem);
    // the copy's work counter runs past the item count by at most one grab
    // per warp and must stay inside 32 bits
    const int64_t nseg = (H / 16 + moe::kCopyPiece - 1) / moe::kCopyPiece;
    const int64_t counter_max =
        T * nseg + static_cast<int64_t>(cap) * moe::kCoopWarps * moe::kCopyGrab;
    if (cap >= nb && counter_max <= static_cast<int64_t>(UINT32_MAX)) {
      moe::CoopScatterArgs sa;
      sa.topk_w = topk_w;
      sa.x = reinterpret_cast<const uint4*>(x);
      sa.x_scale = x_scale;
      sa.ue8m0 = scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR;
      sa.ld_xs = ld_xs;
      sa.H = H;
      sa.xe = reinterpret_cast<uint4*>(xe);
      sa.xe_scale = xe_scale;
      sa.ld_xes = ld_xes;
      sa.row_w = row_w;
      return moe::launch_coop<true>(cap, smem, s, topk_ids, T, K, E, align, d_n_valid, M_cap, nb,
                                    counts, ticket, psum, start, d_total, tile_prefix, m_indices,
                                    src2dst, d_status, sa);
    }
  }
  return layout_then_scatter();
}
