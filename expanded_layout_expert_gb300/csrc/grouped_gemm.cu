// moe_grouped_gemm: FP8 block-scaled grouped GEMM over the expanded rows on
// the 5th-generation tensor cores (the role of DeepGEMM's
// grouped_gemm_nt_f8f8bf16_contig in SGLang moe_runner/deep_gemm.py,
// _run_contiguous_gemm):
//
//   out[r, n] = bf16( sum_kb sA[r, kb] * sW[e, n/128, kb]
//                            * sum_{k in block kb} A[r, k] * W[e, n, k] )
//
// for every row r of expert e's aligned segment. Activations carry one scale
// per 1x128 group, weights one per 128x128 block.
//
// Design (one persistent CTA per SM, warp-specialised):
//  - warp 0, one lane: TMA producer. Per 128-wide K block it loads the
//    128-row A tile and the BN-row W tile (128-byte swizzle) into a ring of
//    shared-memory stages.
//  - warps 1 and 2, one lane each: tcgen05.mma issuers for the even and the
//    odd K blocks (kind::f8f6f4, M=128, N=BN, K=32,
//    4 instructions per K block). Each K block is accumulated into a fresh
//    TMEM buffer (512/BN of them in a ring), because the fp32 block scales
//    cannot be applied inside the tensor core.
//  - warps 4..11: epilogue (two warps per TMEM lane quarter). Each thread
//    owns one row (its TMEM lane) and BN/2 columns; per K block it reads the
//    partial sums with tcgen05.ld, 64 columns per wait, frees the TMEM buffer
//    as soon as its last read has landed, and adds sA * sW * partial into
//    fp32 registers with packed fma.rn.f32x2 ("promotion").
//  - warp 3 is spare; with BN = 256 warpgroup 0 hands its registers to
//    the epilogue warpgroups (setmaxnreg). Scale words are loaded two
//    K blocks before use and decoded only then, so no global load is waited
//    for early. At the end of the tile it converts to bf16 and stores its row
//    (Staged: through shared memory, whole 128-byte rows per instruction; used
//    for short-K GEMMs, where the store is a larger share of a tile).
//  - Fused (moe_grouped_gemm_act_quant): the tile pairs gate and up columns
//    and the epilogue applies silu*mul, the fp8 quantiser and the weight fold
//    instead of storing bf16 (see the kernel's comment).
// The m-tiles come from the layout's per-expert tile prefix, read on the
// device: a CTA maps a linear tile id to (expert, m block, n block), and
// tiles past the device-side total are never visited, so a capacity-sized
// buffer costs nothing beyond its real rows. moe_grouped_gemm sends ue8m0
// scales with N % 256 == 0 to the block-scaled kernel (grouped_gemm_mx.cu).
#include <cuda_bf16.h>

#include <atomic>

#include "act_quant.cuh"
#include "common.cuh"
#include "gemm_host.h"
#include "host_util.h"

#ifndef MOE_GEMM_STAGED_MAX_KB
#define MOE_GEMM_STAGED_MAX_KB 24
#endif
#ifndef MOE_GEMM_STAGES_256
#define MOE_GEMM_STAGES_256 4
#endif

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;      // one scale block along K = one 128-byte swizzle row
constexpr int UMMA_K = 32;   // K of one tcgen05.mma for 8-bit operands
constexpr int kMaxE = 1024;
constexpr int kTraceWords = 8;

template <int BN, bool Staged, bool Fused = false>
struct Cfg {
  static constexpr int kStages = (BN == 256) ? MOE_GEMM_STAGES_256 : 6;
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // Accumulators in flight: TMEM's 512 columns hold 512 / BN of them. More
  // of them hide the round trip from an MMA's completion to the epilogue
  // releasing its buffer.
  static constexpr int kAcc = 512 / BN;
  static constexpr int kEpiWarps = 8;               // two per TMEM lane quarter
  static constexpr int kColsPerWarp = BN / 2;       // columns each epilogue warp promotes
  static constexpr int kFirstEpiWarp = 4;           // warpgroup 0: producer, MMA, 2 spare
  static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
  // BN = 256: 384 threads launch with 168 registers each; warpgroup 0 gives
  // registers to the epilogue warpgroups so each epilogue thread can hold
  // 128 accumulators and a 64-column staging batch (40*128 + 232*256 =
  // 168*384).
  static constexpr bool kRealloc = (BN == 256);
  static constexpr int kRegsLow = 40;
  static constexpr int kRegsHigh = 232;
  static constexpr int kTmemCols = kAcc * BN;
  static constexpr int kNumBars = 2 * kStages + 2 * kAcc + 1 + (Fused ? 4 : 0);
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kTraceOffset = kMiscOffset + 16;          // kTraceWords x u64
  // Fused: row maxima exchanged by the two warps of a lane quarter,
  // [2 tiles][2 halves][128 rows] fp32
  static constexpr int kAmaxOffset = kTraceOffset + kTraceWords * 8;
  static constexpr int kAmaxBytes = Fused ? 2 * 2 * 128 * 4 : 0;
  // Staged: per epilogue warp, 32 rows x 64 bf16 columns go through shared
  // memory for coalesced stores. It pays when tiles are short in K (the
  // store is a larger share of a tile) and costs L1 capacity otherwise (the
  // carve-out leaves less room for the cached activation-scale rows).
  static constexpr int kStoreOffset = (kAmaxOffset + kAmaxBytes + 1023) / 1024 * 1024;
  static constexpr int kStoreBytesPerWarp = Staged ? 32 * 128 : 0;
  // per-expert tables in shared memory when E <= kSmemE (else read from global)
  static constexpr int kTableOffset = kStoreOffset + kEpiWarps * kStoreBytesPerWarp;
  static constexpr int kSmemE = Staged ? 96 : 512;
  static constexpr int kSmemBytes = 1024 + kTableOffset + (2 * kSmemE + 1) * 4;
};

struct Params {
  const void* a_scale;
  int64_t ld_as;
  int ue8m0;
  const void* w_scale;
  const int32_t* start;
  const int32_t* tile_prefix;
  const int32_t* d_total;
  const float* row_w;
  int weight_rows;
  int E, N, Kd;
  int64_t M_cap;
  uint16_t* out;
  int32_t* status;
  unsigned long long* trace;  // optional per-CTA cycle counters
  // Fused gate_up + act+quant: `out` holds down_proj's input codes
  // (uint8 [M_cap, N/2]), `weight_rows` means "fold row_w into the stored
  // scale", and these give the scales (fp32 [M_cap, ld_ds] row-major, or
  // packed ue8m0 int32 words [ceil(N/256/4), ld_ds] written by byte). Reusing
  // fields keeps the parameter block small: a larger one changed the
  // register allocation of the unfused kernels and made them spill.
  void* di_scale;
  int64_t ld_ds;
};

// Bounded wait used while draining: no abort check, only the time limit.
MOE_DEV void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

MOE_DEV uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Trace slots (cycles unless noted), summed per CTA.
enum TraceSlot {
  kTrKernel = 0,      // whole kernel (thread 0)
  kTrProdWait = 1,    // producer waiting for a free stage
  kTrMmaWaitTmem = 2, // MMA issuers waiting for a free TMEM buffer (summed)
  kTrMmaWaitData = 3, // MMA issuers waiting for TMA data (summed)
  kTrEpiWait = 4,     // unused (zero): timing the epilogue's waits slowed it
  kTrEpiTile = 5,     // epilogue warp 4: tile-end work (store, or act+quant)
  kTrUnused6 = 6,
  kTrKBlocks = 7,     // K blocks this CTA processed (count)
};

// Fused (BN = 256 only): gate_up with silu(gate)*up and the fp8 quantiser of
// down_proj's input in the epilogue (W = W13 [E, 2I, H]). A tile is 128 rows
// x 128 intermediate columns t*128..: its B tile stacks W13's gate rows
// [t*128, +128) over its up rows [I + t*128, +128), so each output group of
// 128 sits in one accumulator (gate columns 0-127, up 128-255). Each
// epilogue warp promotes gate columns [64 half, +64) with the gate block's
// weight scale and up columns [128 + 64 half, +64) with the up block's, then
// forms h = bf16(silu(bf16 g) * bf16 u), exchanges its row maximum with the
// other warp of its lane quarter, and writes codes and the group's scale.
// The arithmetic is that of the stand-alone launches, bit for bit.
//
// Ue8m0 fixes the scale format at compile time (p.ue8m0 says the same at run
// time): the per-K-block scale loads and decode are in the epilogue's inner
// loop, and selecting between the two formats there cost 5-9 % of the
// kernel's time.
template <int BN, bool Staged, bool Fused, bool Ue8m0>
__global__ void __launch_bounds__(Cfg<BN, Staged, Fused>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const Params p) {
  using C = Cfg<BN, Staged, Fused>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + C::kAcc;
  uint64_t* mma_done = tempty + C::kAcc;
  uint64_t* amax_bar = mma_done + 1;  // Fused: [4], one per TMEM lane quarter
  float* s_amax = reinterpret_cast<float*>(smem + C::kAmaxOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOffset + 4);
  unsigned long long* s_trace = reinterpret_cast<unsigned long long*>(smem + C::kTraceOffset);
  // per-expert tables: shared memory for up to kSmemE experts, else global
  const bool smem_tables = p.E <= C::kSmemE;
  int* t_tp = reinterpret_cast<int*>(smem + C::kTableOffset);
  int* t_start = t_tp + (p.E + 1);
  const int* s_tp = smem_tables ? t_tp : p.tile_prefix;
  const int* s_start = smem_tables ? t_start : p.start;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool tracing = p.trace != nullptr;
  const long long t_kernel0 = clock64();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < C::kAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], C::kEpiWarps);
    }
    mbar_init(mma_done, 2);  // one commit per MMA issuer
    if (Fused)
      for (int q = 0; q < 4; ++q) mbar_init(&amax_bar[q], 64);  // both warps of the quarter
    *abort_flag = 0;
    for (int i = 0; i < kTraceWords; ++i) s_trace[i] = 0ull;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (smem_tables) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) t_tp[i] = p.tile_prefix[i];
    for (int i = threadIdx.x; i < p.E; i += blockDim.x) t_start[i] = p.start[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int total = *p.d_total;
  if (total > p.M_cap) total = static_cast<int>(p.M_cap);
  // tiles per m block: BN output columns, or (fused) 128 intermediate columns
  const int num_n = Fused ? p.N / 256 : p.N / BN;
  const int I = p.N / 2;
  const int num_tiles = s_tp[p.E] * num_n;
  const int KB = p.Kd / BK;
  const int NB = p.N / 128;

  // linear tile -> expert, first row, rows in this tile
  auto tile_rows = [&](int tile, int& e, int& row0, int& rows) {
    const int m = tile / num_n;
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tp[mid] <= m) lo = mid; else hi = mid - 1;
    }
    e = lo;
    row0 = s_start[e] + (m - s_tp[e]) * BM;
    const int seg_end = (e + 1 < p.E) ? min(s_start[e + 1], total) : total;
    rows = min(BM, seg_end - row0);
  };

  if (warp < C::kFirstEpiWarp) {
    // Warpgroup 0; with BN = 256 it hands registers to the epilogue (each
    // role's branch starts with its own setmaxnreg so the register allocator
    // sees the limit that holds in it).
    if constexpr (C::kRealloc) regs_release<C::kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      unsigned long long t_wait = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int e, row0, rows;
        tile_rows(tile, e, row0, rows);
        const int n0 = (tile % num_n) * BN;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const long long t0 = tracing ? clock64() : 0;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          if (tracing) t_wait += clock64() - t0;
          uint8_t* sa = smem + stage * C::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          tma_load_2d(sa, &tmA, kb * BK, row0, &full[stage]);
          if (Fused) {
            const int t = tile % num_n;
            tma_load_2d(sa + C::kABytes, &tmB, kb * BK, e * p.N + t * 128, &full[stage]);
            tma_load_2d(sa + C::kABytes + C::kBBytes / 2, &tmB, kb * BK, e * p.N + I + t * 128,
                        &full[stage]);
          } else {
            tma_load_2d(sa + C::kABytes, &tmB, kb * BK, e * p.N + n0, &full[stage]);
          }
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (tracing) s_trace[kTrProdWait] = t_wait;
      // Let the last loads land before the CTA can exit.
      const int outstanding = issued < C::kStages ? issued : C::kStages;
      for (int i = 1; i <= outstanding; ++i) {
        int s = stage - i;
        uint32_t ph = phase;
        if (s < 0) { s += C::kStages; ph ^= 1u; }
        drain_wait(&full[s], ph);
      }
    } else if ((warp == 1 || warp == 2) && lane == 0) {
      // ---------------------------------------------------------- MMA issuers
      // Two threads issue the MMAs: warp 1 the even K blocks of the CTA's
      // running count, warp 2 the odd ones, each with its own accumulator
      // buffer when there are two. An MMA issue blocks while the tensor
      // pipe's queue is full, so with one thread the pipe drains while that
      // thread waits on its two barriers; with two, one waits while the
      // other issues. K blocks are independent (own accumulator, own stage),
      // so the order in which the pipe takes them changes no result.
      constexpr uint32_t idesc = idesc_f8_f32(BM, BN);
      const int par = warp - 1;
      unsigned long long t_tmem = 0, t_data = 0, nkb = 0;
      long long g = 0;  // the CTA's running K-block count
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++g) {
          if (static_cast<int>(g & 1) != par) continue;
          const int stage = static_cast<int>(g % C::kStages);
          const uint32_t phase = static_cast<uint32_t>((g / C::kStages) & 1);
          const int acc = static_cast<int>(g % C::kAcc);
          const uint32_t acc_phase = static_cast<uint32_t>((g / C::kAcc) & 1);
          const long long t0 = tracing ? clock64() : 0;
          if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          const long long t1 = tracing ? clock64() : 0;
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          if (tracing) {
            const long long t2 = clock64();
            t_tmem += t1 - t0;
            t_data += t2 - t1;
            ++nkb;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            tc_mma_f8(d, sw128_kmajor_desc(sa + k * UMMA_K), sw128_kmajor_desc(sb + k * UMMA_K),
                      idesc, k > 0 ? 1u : 0u);
          tc_commit(&empty[stage]);
          tc_commit(&tfull[acc]);
        }
      }
      if (tracing) {  // summed over both issuers
        atomicAdd(&s_trace[kTrMmaWaitTmem], t_tmem);
        atomicAdd(&s_trace[kTrMmaWaitData], t_data);
        atomicAdd(&s_trace[kTrKBlocks], nkb);
      }
      // Every MMA issued so far must complete before TMEM is released
      // (mma_done counts one arrival per issuer).
      tc_commit(mma_done);
      drain_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if constexpr (C::kRealloc) regs_claim<C::kRegsHigh>();
    const int ew = warp - C::kFirstEpiWarp;
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int half = ew >> 2;      // which half of the BN columns
    const int row_in_tile = quarter * 32 + lane;
    const uint8_t* ws8 = static_cast<const uint8_t*>(p.w_scale);
    const float* wsf = static_cast<const float*>(p.w_scale);
    int acc_buf = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int iter = 0;
    unsigned long long t_epi_wait = 0, t_epi_tile = 0;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++iter) {
      int e, row0, rows;
      tile_rows(tile, e, row0, rows);
      const int n_tile = tile % num_n;
      const int col0 = n_tile * BN + half * C::kColsPerWarp;  // this warp's first column
      const int row = row0 + row_in_tile;
      const bool row_ok = row_in_tile < rows && row < p.M_cap;
      // weight-scale rows of this warp's two 64-column batches: the same
      // 128-column block, or (fused) the gate block and the up block
      const int nb0 = Fused ? n_tile : col0 / 128;
      const int nb1 = Fused ? I / 128 + n_tile : nb0;
      const int64_t wbase = (static_cast<int64_t>(e) * NB + nb0) * KB;
      const int64_t wbase1 = (static_cast<int64_t>(e) * NB + nb1) * KB;

      // Raw scale words, loaded two K blocks before they are used and only
      // decoded (and multiplied) then, so no load is waited for early.
      const float* asf = static_cast<const float*>(p.a_scale);
      const uint32_t* asw = static_cast<const uint32_t*>(p.a_scale);
      auto load_raw = [&](int kb, uint32_t& ra, uint32_t& rw, uint32_t& rw1) {
        if (kb >= KB) {
          ra = 0u;
          rw = 0u;
          rw1 = 0u;
          return;
        }
        rw = Ue8m0 ? static_cast<uint32_t>(ws8[wbase + kb]) : __float_as_uint(wsf[wbase + kb]);
        if (Fused)
          rw1 = Ue8m0 ? static_cast<uint32_t>(ws8[wbase1 + kb]) : __float_as_uint(wsf[wbase1 + kb]);
        ra = 0u;
        if (row_ok)
          ra = Ue8m0 ? asw[static_cast<int64_t>(kb >> 2) * p.ld_as + row]
                       : __float_as_uint(asf[static_cast<int64_t>(row) * p.ld_as + kb]);
      };
      auto decode = [&](int kb, uint32_t ra, uint32_t rw) -> float {
        if (Ue8m0) return ue8m0_to_f32((ra >> (8 * (kb & 3))) & 0xFFu) * ue8m0_to_f32(rw);
        return __uint_as_float(ra) * __uint_as_float(rw);
      };

      // Accumulators as packed pairs: one fma.rn.f32x2 promotes two columns.
      float2 acc[C::kColsPerWarp / 2];
#pragma unroll
      for (int j = 0; j < C::kColsPerWarp / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);

      // One K block: wait for its accumulator, read it from TMEM 16 columns
      // at a time, fold it in with the block's scale, free the buffer as
      // soon as the last read has landed.
      auto kblock = [&](int kb, uint32_t& ra, uint32_t& rw, uint32_t& rw1) {
        if (!ok || kb >= KB) return;
        // all lanes leave together: the TMEM loads below are warp-collective
        const bool got = mbar_wait_warp(&tfull[acc_buf], acc_phase, abort_flag, p.status);
        if (!got) {
          ok = false;
          return;
        }
        tc_fence_after();
        const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                            static_cast<uint32_t>(acc_buf * BN);
        // 64 columns per wait; the buffer is released right after the last
        // read, before that batch is promoted, so the MMA can reuse it as
        // early as possible.
        constexpr int kBatches = C::kColsPerWarp / 64;
        float sc0 = 0.0f, sc1 = 0.0f;
#pragma unroll
        for (int bt = 0; bt < kBatches; ++bt) {
          const uint32_t bcol = Fused ? static_cast<uint32_t>(bt * 128 + half * 64)
                                      : static_cast<uint32_t>(half * C::kColsPerWarp + bt * 64);
          uint32_t va[32], vb[32];
          tc_ld32(tq + bcol, va);
          tc_ld32(tq + bcol + 32, vb);
          if (bt == 0) {
            // decode this K block's scales and fetch those of K block kb + 2
            // while the first TMEM load is in flight
            sc0 = decode(kb, ra, rw);
            sc1 = Fused ? decode(kb, ra, rw1) : sc0;
            load_raw(kb + 2, ra, rw, rw1);
          }
          const float2 sc = bt == 0 ? make_float2(sc0, sc0) : make_float2(sc1, sc1);
          tc_wait64(va, vb);
          if (bt == kBatches - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc_buf]);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)
            acc[bt * 32 + j] = __ffma2_rn(sc, make_float2(__uint_as_float(va[2 * j]),
                                                          __uint_as_float(va[2 * j + 1])),
                                          acc[bt * 32 + j]);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            acc[bt * 32 + 16 + j] = __ffma2_rn(sc, make_float2(__uint_as_float(vb[2 * j]),
                                                               __uint_as_float(vb[2 * j + 1])),
                                               acc[bt * 32 + 16 + j]);
        }
        if (++acc_buf == C::kAcc) {
          acc_buf = 0;
          acc_phase ^= 1u;
        }
      };

      uint32_t ra0, rw0, rx0, ra1, rw1, rx1;
      load_raw(0, ra0, rw0, rx0);
      load_raw(1, ra1, rw1, rx1);
      for (int kb0 = 0; kb0 < KB && ok; kb0 += 2) {
        kblock(kb0 + 0, ra0, rw0, rx0);
        kblock(kb0 + 1, ra1, rw1, rx1);
      }
      if (!ok) break;
      const long long tt0 = tracing ? clock64() : 0;
      if constexpr (Fused) {
        // h = bf16(silu(bf16 g) * bf16 u): gate pairs acc[0..31], up acc[32..63]
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float hx = silu_mul_bf16(bf16_round(acc[j].x), bf16_round(acc[32 + j].x));
          const float hy = silu_mul_bf16(bf16_round(acc[j].y), bf16_round(acc[32 + j].y));
          acc[j] = make_float2(hx, hy);
          m = fmaxf(m, fmaxf(fabsf(hx), fabsf(hy)));
        }
        // the other warp's maximum for the same row (double-buffered by tile)
        const int par = iter & 1;
        s_amax[(par * 2 + half) * 128 + row_in_tile] = m;
        mbar_arrive(&amax_bar[quarter]);
        const bool got = mbar_wait_warp(&amax_bar[quarter], static_cast<uint32_t>(par),
                                        abort_flag, p.status);
        if (!got) break;
        const float amax = fmaxf(m, s_amax[(par * 2 + (half ^ 1)) * 128 + row_in_tile]);
        float sc, inv;
        uint32_t bexp;
        group_scale(amax, Ue8m0, sc, inv, bexp);
        if (row_ok) {
          uint8_t* di = reinterpret_cast<uint8_t*>(p.out);
          uint4* dst = reinterpret_cast<uint4*>(di + static_cast<int64_t>(row) * I +
                                                n_tile * 128 + half * 64);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float h[16] = {acc[8 * q + 0].x, acc[8 * q + 0].y, acc[8 * q + 1].x,
                                 acc[8 * q + 1].y, acc[8 * q + 2].x, acc[8 * q + 2].y,
                                 acc[8 * q + 3].x, acc[8 * q + 3].y, acc[8 * q + 4].x,
                                 acc[8 * q + 4].y, acc[8 * q + 5].x, acc[8 * q + 5].y,
                                 acc[8 * q + 6].x, acc[8 * q + 6].y, acc[8 * q + 7].x,
                                 acc[8 * q + 7].y};
            const uint2 lo = fp8x8(h, inv), hi = fp8x8(h + 8, inv);
            dst[q] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
          if (half == 0) {
            if (Ue8m0) {
              // byte t%4 of word (t/4, row); the last group also clears the
              // word's unused bytes
              uint8_t* w = static_cast<uint8_t*>(p.di_scale) +
                           (static_cast<int64_t>(n_tile >> 2) * p.ld_ds + row) * 4;
              w[n_tile & 3] = static_cast<uint8_t>(bexp);
              if (n_tile == num_n - 1)
                for (int z = (n_tile & 3) + 1; z < 4; ++z) w[z] = 0;
            } else {
              const float wgt = p.weight_rows ? p.row_w[row] : 1.0f;
              static_cast<float*>(p.di_scale)[static_cast<int64_t>(row) * p.ld_ds + n_tile] =
                  __fmul_rn(sc, wgt);
            }
          }
        }
      } else if constexpr (Staged) {
      // Store through shared memory: each thread writes its row's 64-column
      // slices (swizzled, conflict-free), then the warp writes 4 rows of 128
      // contiguous bytes per instruction.
      {
        const float wm = (p.weight_rows && row_ok) ? p.row_w[row] : 1.0f;
        uint8_t* stg = smem + C::kStoreOffset + ew * C::kStoreBytesPerWarp;
        const uint32_t stg_s = smem_u32(stg);
        const int row_w0 = row0 + quarter * 32;          // this warp's first row
        const int rows_w = rows - quarter * 32;          // valid rows of this warp
#pragma unroll
        for (int ps = 0; ps < C::kColsPerWarp / 64; ++ps) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float2* a2 = &acc[ps * 32 + c * 4];
            const uint32_t x0 = pack_bf16x2(a2[0].x * wm, a2[0].y * wm);
            const uint32_t x1 = pack_bf16x2(a2[1].x * wm, a2[1].y * wm);
            const uint32_t x2 = pack_bf16x2(a2[2].x * wm, a2[2].y * wm);
            const uint32_t x3 = pack_bf16x2(a2[3].x * wm, a2[3].y * wm);
            const uint32_t off = static_cast<uint32_t>(lane * 128 + ((c ^ (lane & 7)) << 4));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg_s + off), "r"(x0),
                         "r"(x1), "r"(x2), "r"(x3)
                         : "memory");
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3);
            const int c = lane & 7;
            uint4 v;
            const uint32_t off = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(stg_s + off)
                         : "memory");
            const int grow = row_w0 + r;
            if (r < rows_w && grow < p.M_cap)
              *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(grow) * p.N + col0 + ps * 64 +
                                        c * 8) = v;
          }
          __syncwarp();
        }
      }
      } else {
        if (row_ok) {
          const float wm = p.weight_rows ? p.row_w[row] : 1.0f;
          uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.N + col0);
#pragma unroll
          for (int v = 0; v < C::kColsPerWarp / 8; ++v) {
            uint4 o;
            o.x = pack_bf16x2(acc[v * 4 + 0].x * wm, acc[v * 4 + 0].y * wm);
            o.y = pack_bf16x2(acc[v * 4 + 1].x * wm, acc[v * 4 + 1].y * wm);
            o.z = pack_bf16x2(acc[v * 4 + 2].x * wm, acc[v * 4 + 2].y * wm);
            o.w = pack_bf16x2(acc[v * 4 + 3].x * wm, acc[v * 4 + 3].y * wm);
            dst[v] = o;
          }
        }
      }
      if (tracing) t_epi_tile += clock64() - tt0;
    }
    if (tracing && ew == 0 && lane == 0) {
      s_trace[kTrEpiWait] = t_epi_wait;
      s_trace[kTrEpiTile] = t_epi_tile;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (tracing && threadIdx.x == 0) {
    s_trace[kTrKernel] = static_cast<unsigned long long>(clock64() - t_kernel0);
    for (int i = 0; i < kTraceWords; ++i) p.trace[blockIdx.x * kTraceWords + i] = s_trace[i];
  }
}


std::atomic<unsigned long long*> g_trace{nullptr};

template <int BN, bool Staged, bool Fused, bool Ue8m0>
int launch_fmt(const CUtensorMap& ta, const CUtensorMap& tb, const Params& prm, cudaStream_t s) {
  using C = Cfg<BN, Staged, Fused>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(grouped_gemm_kernel<BN, Staged, Fused, Ue8m0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return check_launch("cudaFuncSetAttribute(grouped_gemm_kernel)");
    attr_set[dev] = true;
  }
  grouped_gemm_kernel<BN, Staged, Fused, Ue8m0>
      <<<device_sm_count(), C::kThreads, C::kSmemBytes, s>>>(ta, tb, prm);
  return check_launch("grouped_gemm_kernel");
}

template <int BN, bool Staged, bool Fused = false>
int launch(const CUtensorMap& ta, const CUtensorMap& tb, const Params& prm, cudaStream_t s) {
  return prm.ue8m0 ? launch_fmt<BN, Staged, Fused, true>(ta, tb, prm, s)
                   : launch_fmt<BN, Staged, Fused, false>(ta, tb, prm, s);
}

}  // namespace
}  // namespace moe

extern "C" int moe_gemm_set_trace(uint64_t* d_trace) {
  moe::g_trace.store(reinterpret_cast<unsigned long long*>(d_trace));
  return MOE_OK;
}

extern "C" int moe_grouped_gemm(const uint8_t* A, const void* A_scale, int scale_layout,
                                int64_t ld_as, const int32_t* start, const int32_t* tile_prefix,
                                const int32_t* d_total, const uint8_t* W, const void* W_scale,
                                const float* row_w, int flags, int E, int N, int Kd,
                                int64_t M_cap, uint16_t* out, int32_t* d_status,
                                moe_stream_t stream) {
  MOE_REQUIRE(A && A_scale && start && tile_prefix && d_total && W && W_scale && out,
              "moe_grouped_gemm: null pointer");
  MOE_REQUIRE(E > 0 && E <= moe::kMaxE, "moe_grouped_gemm: E must be in [1, 1024]");
  MOE_REQUIRE(N > 0 && N % 128 == 0 && Kd > 0 && Kd % 128 == 0,
              "moe_grouped_gemm: N and Kd must be positive multiples of 128");
  MOE_REQUIRE(M_cap > 0 && M_cap <= INT32_MAX && static_cast<int64_t>(E) * N <= INT32_MAX,
              "moe_grouped_gemm: sizes exceed int32");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_grouped_gemm: bad scale layout");
  if (scale_layout == MOE_SCALE_F32_ROWMAJOR) {
    MOE_REQUIRE(ld_as >= Kd / 128, "moe_grouped_gemm: scale leading dimension < Kd/128");
  } else {
    MOE_REQUIRE(ld_as >= M_cap, "moe_grouped_gemm: packed scale leading dimension < M_cap");
  }
  MOE_REQUIRE(!(flags & MOE_WEIGHT_OUTPUT_ROWS) || row_w, "moe_grouped_gemm: row weighting needs row_w");
  MOE_REQUIRE(moe::aligned(A, 16) && moe::aligned(W, 16) && moe::aligned(out, 16),
              "moe_grouped_gemm: A, W and out must be 16-byte aligned");
  MOE_REQUIRE_DEVICE();

  // Power-of-two scales go to the tensor core's block scaling.
  const bool block_scaled = scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR && N % 256 == 0 &&
                            !(flags & (MOE_GEMM_TILE_N128 | MOE_GEMM_PER_KBLOCK_PROMOTION));
  if (block_scaled) {
    moe::MxGemmArgs a;
    a.A = A;
    a.A_scale = static_cast<const uint32_t*>(A_scale);
    a.ld_as = ld_as;
    a.start = start;
    a.tile_prefix = tile_prefix;
    a.d_total = d_total;
    a.W = W;
    a.W_scale = static_cast<const uint8_t*>(W_scale);
    a.row_w = (flags & MOE_WEIGHT_OUTPUT_ROWS) ? row_w : nullptr;
    a.E = E;
    a.N = N;
    a.Kd = Kd;
    a.M_cap = M_cap;
    a.out = out;
    a.status = d_status;
    a.trace = moe::g_trace.load();
    return moe::launch_grouped_gemm_mx(a, reinterpret_cast<cudaStream_t>(stream));
  }
  const int BN = (N % 256 == 0 && !(flags & MOE_GEMM_TILE_N128)) ? 256 : 128;
  CUtensorMap ta, tb;
  int rc = moe::make_tmap_k128(&ta, A, Kd, M_cap, Kd, moe::BM);
  if (rc != MOE_OK) return rc;
  rc = moe::make_tmap_k128(&tb, W, Kd, static_cast<uint64_t>(E) * N, Kd, BN);
  if (rc != MOE_OK) return rc;
  moe::Params prm;
  prm.a_scale = A_scale;
  prm.ld_as = ld_as;
  prm.ue8m0 = scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR;
  prm.w_scale = W_scale;
  prm.start = start;
  prm.tile_prefix = tile_prefix;
  prm.d_total = d_total;
  prm.row_w = row_w;
  prm.weight_rows = (flags & MOE_WEIGHT_OUTPUT_ROWS) ? 1 : 0;
  prm.E = E;
  prm.N = N;
  prm.Kd = Kd;
  prm.M_cap = M_cap;
  prm.out = out;
  prm.status = d_status;
  prm.trace = moe::g_trace.load();
  prm.di_scale = nullptr;
  prm.ld_ds = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Short-K GEMMs (down_proj) spend a larger share of each tile on the
  // store, so they take the staged store; long-K ones keep the L1 room.
  const bool staged = (Kd / 128) <= MOE_GEMM_STAGED_MAX_KB;
  if (BN == 256)
    return staged ? moe::launch<256, true>(ta, tb, prm, s) : moe::launch<256, false>(ta, tb, prm, s);
  return staged ? moe::launch<128, true>(ta, tb, prm, s) : moe::launch<128, false>(ta, tb, prm, s);
}

extern "C" int moe_grouped_gemm_act_quant(const uint8_t* A, const void* A_scale, int scale_layout,
                                          int64_t ld_as, const int32_t* start,
                                          const int32_t* tile_prefix, const int32_t* d_total,
                                          const uint8_t* W13, const void* W13_scale,
                                          const float* row_w, int flags, int E, int I, int H,
                                          int64_t M_cap, uint8_t* di, void* di_scale,
                                          int64_t ld_ds, int32_t* d_status, moe_stream_t stream) {
  MOE_REQUIRE(A && A_scale && start && tile_prefix && d_total && W13 && W13_scale && di && di_scale,
              "moe_grouped_gemm_act_quant: null pointer");
  MOE_REQUIRE(E > 0 && E <= moe::kMaxE, "moe_grouped_gemm_act_quant: E must be in [1, 1024]");
  MOE_REQUIRE(I > 0 && I % 128 == 0 && H > 0 && H % 128 == 0,
              "moe_grouped_gemm_act_quant: I and H must be positive multiples of 128");
  MOE_REQUIRE(M_cap > 0 && M_cap <= INT32_MAX && static_cast<int64_t>(E) * 2 * I <= INT32_MAX,
              "moe_grouped_gemm_act_quant: sizes exceed int32");
  MOE_REQUIRE(scale_layout == MOE_SCALE_F32_ROWMAJOR || scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR,
              "moe_grouped_gemm_act_quant: bad scale layout");
  const bool ue8m0 = scale_layout == MOE_SCALE_UE8M0_PACKED_COLMAJOR;
  const bool fold = (flags & MOE_FOLD_WEIGHT_INTO_SCALE) != 0;
  MOE_REQUIRE(!fold || (!ue8m0 && row_w),
              "moe_grouped_gemm_act_quant: the fold needs row_w and fp32 scales");
  if (ue8m0) {
    MOE_REQUIRE(ld_as >= M_cap && ld_ds >= M_cap,
                "moe_grouped_gemm_act_quant: packed scale leading dimension < M_cap");
  } else {
    MOE_REQUIRE(ld_as >= H / 128 && ld_ds >= I / 128,
                "moe_grouped_gemm_act_quant: scale leading dimension too small");
  }
  MOE_REQUIRE(moe::aligned(A, 16) && moe::aligned(W13, 16) && moe::aligned(di, 16) &&
                  moe::aligned(di_scale, 4),
              "moe_grouped_gemm_act_quant: A, W13 and di must be 16-byte aligned");
  MOE_REQUIRE_DEVICE();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!ue8m0 || (flags & MOE_GEMM_PER_KBLOCK_PROMOTION)) {
    // fp32 scales: per-K-block promotion kernel with the fused epilogue
    CUtensorMap ta, tb;
    int rc = moe::make_tmap_k128(&ta, A, H, M_cap, H, moe::BM);
    if (rc != MOE_OK) return rc;
    rc = moe::make_tmap_k128(&tb, W13, H, static_cast<uint64_t>(E) * 2 * I, H, 128);
    if (rc != MOE_OK) return rc;
    moe::Params prm;
    prm.a_scale = A_scale;
    prm.ld_as = ld_as;
    prm.ue8m0 = ue8m0 ? 1 : 0;
    prm.w_scale = W13_scale;
    prm.start = start;
    prm.tile_prefix = tile_prefix;
    prm.d_total = d_total;
    prm.row_w = row_w;
    prm.weight_rows = fold ? 1 : 0;  // fused: fold the weight into the stored scale
    prm.E = E;
    prm.N = 2 * I;
    prm.Kd = H;
    prm.M_cap = M_cap;
    prm.out = reinterpret_cast<uint16_t*>(di);  // fused: the fp8 codes
    prm.status = d_status;
    prm.trace = moe::g_trace.load();
    prm.di_scale = di_scale;
    prm.ld_ds = ld_ds;
    return moe::launch<256, false, true>(ta, tb, prm, s);
  }
  moe::MxGemmArgs a;
  a.A = A;
  a.A_scale = static_cast<const uint32_t*>(A_scale);
  a.ld_as = ld_as;
  a.start = start;
  a.tile_prefix = tile_prefix;
  a.d_total = d_total;
  a.W = W13;
  a.W_scale = static_cast<const uint8_t*>(W13_scale);
  a.row_w = nullptr;
  a.E = E;
  a.N = 2 * I;
  a.Kd = H;
  a.M_cap = M_cap;
  a.out = nullptr;
  a.status = d_status;
  a.trace = moe::g_trace.load();
  a.di = di;
  a.di_scale = static_cast<uint8_t*>(di_scale);
  a.ld_ds = ld_ds;
  return moe::launch_grouped_gemm_mx(a, s);
}
