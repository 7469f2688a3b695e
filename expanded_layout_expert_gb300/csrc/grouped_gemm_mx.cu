// Block-scaled grouped GEMM for power-of-two (ue8m0) scales: the scales are
// applied inside the tensor core (tcgen05.mma kind::mxf8f6f4.block_scale), so
// a tile accumulates its whole K range in one TMEM accumulator and the
// epilogue runs once per tile instead of once per K block.
//
//   out[r, n] = bf16( w_r * sum_kb 2^(a[r,kb]-127) * 2^(b[e,n/128,kb]-127)
//                               * sum_{k in block kb} A[r, k] * W[e, n, k] )
//
// with w_r = row_w[r] on the weighted-output path and 1 otherwise (the ue8m0
// path of the expanded MoE layer: SGLang moe_runner/deep_gemm.py,
// DeepGemmMoeQuantInfo with ue8m0 scales; the per-row output weighting of
// SGLang PR 20096, "apply topk weights to down_output").
//
// Each 128-wide K block carries one activation scale per row and one weight
// scale per 128 output columns. The tensor core takes one ue8m0 scale per row
// of A and of B for every K = 32 step, so the four steps of a K block simply
// reuse the block's scale; a 32-bit scale word packs four K blocks and the
// instruction descriptor selects the byte.
//
// Roles (one persistent CTA per SM, 384 threads):
//  - warp 0, one lane: TMA producer of the A (128 x 128 B) and W (256 x
//    128 B) tiles, 128-byte swizzle, into a ring of shared-memory stages.
//  - warp 2: scale loader. Per group of four K blocks it reads the tile's
//    128 packed activation-scale words (coalesced) and the two weight-scale
//    words, and writes them to a shared-memory slot in the order the
//    32-lane TMEM copy expects: the 16 bytes of lane i hold the words of
//    rows i, i+32, i+64, i+96 (so TMEM column j of lane i is row i + 32 j).
//  - warp 1, one lane: MMA issuer. At the start of each group it copies the
//    slot into TMEM (tcgen05.cp 32x128b.warpx4, ordered before the MMAs that
//    read it), then issues four K = 32 block-scaled MMAs per K block into
//    the tile's accumulator.
//  - warps 4..11: epilogue. Two warps per TMEM lane quarter, 128 columns
//    each: read the finished accumulator (4 x 32 columns, one wait), free it
//    for the next tile, scale by the row weight, convert to bf16 and store.
// TMEM: columns 0-255 the accumulator, 256 + 16 s the scale slot s
// (A: 4 columns, B: 8 columns).
#include <cuda_bf16.h>

#include "act_quant.cuh"
#include "common.cuh"
#include "gemm_host.h"
#include "host_util.h"

namespace moe {
namespace {

namespace mx {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int UMMA_K = 32;
constexpr int kMaxE = 1024;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK;
constexpr int kBBytes = BN * BK;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSfSlots = 4;              // groups of four K blocks in flight
constexpr int kSfBytesA = 32 * 16;       // 128 rows, one word each
constexpr int kSfBytesB = 2 * 32 * 16;   // 256 columns, one word each
constexpr int kSfSlotBytes = kSfBytesA + kSfBytesB;
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 4;
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kTmemCols = 512;
constexpr int kSfCol = 256;
constexpr int kSfSlotCols = 16;

constexpr int kSfOffset = kStages * kStageBytes;
constexpr int kBarOffset = kSfOffset + kSfSlots * kSfSlotBytes;
constexpr int kNumBars = 2 * kStages + 2 * kSfSlots + 3 + 4;  // + 4 amax exchanges
constexpr int kMiscOffset = kBarOffset + kNumBars * 8;   // tmem slot, abort flag
constexpr int kTraceOffset = kMiscOffset + 16;           // kTraceWords x u64
constexpr int kAmaxOffset = kTraceOffset + 8 * 8;        // fused: [2 tiles][2 halves][128 rows] f32
constexpr int kTableOffset = kAmaxOffset + 2 * 2 * 128 * 4;  // tile prefix (E+1), start (E)
constexpr int kSmemBytes = 1024 + kTableOffset + (2 * kMaxE + 1) * 4;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kSfCol + kSfSlots * kSfSlotCols <= kTmemCols, "TMEM budget");

struct Params {
  const uint32_t* a_scale;
  int64_t ld_as;
  const uint8_t* w_scale;
  const int32_t* start;
  const int32_t* tile_prefix;
  const int32_t* d_total;
  const float* row_w;
  int E, N, Kd;
  int64_t M_cap;
  uint16_t* out;
  int32_t* status;
  unsigned long long* trace;  // optional: 8 cycle counters per CTA
  // fused gate_up + act+quant: down_proj's input codes [M_cap, N/2] and
  // packed ue8m0 scales (bytes of int32 words [ceil(N/256/4), ld_ds])
  uint8_t* di;
  uint8_t* di_scale;
  int64_t ld_ds;
};

// Trace words (cycles, summed per CTA): whole kernel, producer waiting for a
// free stage, MMA waiting for the accumulator, for operands, for scales,
// epilogue warp 4 waiting for a finished tile, its work per tile, K blocks.
constexpr int kTraceWords = 8;

MOE_DEV void drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

MOE_DEV uint32_t bf16x2_bits(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// kTrace: a separate instantiation carries the cycle counters, so the
// production kernel has none of their code.
// kFused: gate_up with silu(gate)*up and the fp8 quantiser of down_proj's
// input in the epilogue (W = W13 [E, 2I, H]). A tile is 128 rows x 128
// intermediate columns t*128..: its B tile stacks W13's gate rows
// [t*128, +128) over its up rows [I + t*128, +128), so every output group of
// 128 sits in one accumulator (gate in columns 0-127, up in 128-255). The
// two epilogue warps of a lane quarter take 64 columns each, exchange their
// row maxima through shared memory, and write the codes and the group's
// scale byte; gate_up's bf16 output never goes to memory. The arithmetic is
// the stand-alone kernels' (bf16 rounding of the GEMM output, then the
// shared act+quant math), so the codes and scales are the same bit for bit.
template <bool kTrace, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);
  uint64_t* empty = full + kStages;
  uint64_t* sf_full = empty + kStages;
  uint64_t* sf_empty = sf_full + kSfSlots;
  uint64_t* tfull = sf_empty + kSfSlots;
  uint64_t* tempty = tfull + 1;
  uint64_t* mma_done = tempty + 1;
  uint64_t* amax_bar = mma_done + 1;  // [4], one per TMEM lane quarter
  float* s_amax = reinterpret_cast<float*>(smem + kAmaxOffset);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOffset + 4);
  unsigned long long* s_trace = reinterpret_cast<unsigned long long*>(smem + kTraceOffset);
  int* s_tp = reinterpret_cast<int*>(smem + kTableOffset);
  int* s_start = s_tp + (p.E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr bool tracing = kTrace;
  const long long t_kernel0 = tracing ? clock64() : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSfSlots; ++s) {
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    mbar_init(mma_done, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&amax_bar[q], 2);  // lane 0 of both warps of the quarter
    *abort_flag = 0;
    for (int i = 0; i < kTraceWords; ++i) s_trace[i] = 0ull;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_tp[i] = p.tile_prefix[i];
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) s_start[i] = p.start[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int total = *p.d_total;
  if (total > p.M_cap) total = static_cast<int>(p.M_cap);
  // tiles per m block: 256 output columns, or (fused) 128 intermediate columns
  const int num_n = kFused ? p.N / 256 : p.N / BN;
  const int I = p.N / 2;
  const int num_tiles = s_tp[p.E] * num_n;
  const int KB = p.Kd / BK;
  const int NB = p.N / 128;

  // Tiles go expert by expert. Inside an expert the fused gate_up goes n
  // tile by n tile (the expert's m blocks for its first n tile, then for
  // its second, ...): the CTAs that read one weight tile hold consecutive
  // tile ids and run it at the same time, so an expert's W13 (29 MB at
  // H = 7168, I = 2048) need not stay in L2 from one wave of tiles to the
  // next; only its activation rows do. The down GEMM (W2 half that size,
  // more n tiles) keeps the m-major order, which measured faster there.
  auto tile_coords = [&](int tile, int& e, int& row0, int& rows, int& nt) {
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tp[mid] * num_n <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int j = tile - s_tp[e] * num_n;
    int m_local;
    if constexpr (kFused) {
      const int mb = s_tp[e + 1] - s_tp[e];  // > 0: the expert owns the tile
      nt = j / mb;
      m_local = j - nt * mb;
    } else {
      m_local = j / num_n;
      nt = j - m_local * num_n;
    }
    row0 = s_start[e] + m_local * BM;
    const int seg_end = (e + 1 < p.E) ? min(s_start[e + 1], total) : total;
    rows = min(BM, seg_end - row0);
  };

  const int KG = (KB + 3) / 4;  // groups of four K blocks (one packed scale word)

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      unsigned long long t_wait = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int e, row0, rows, nt;
        tile_coords(tile, e, row0, rows, nt);
        const int n0 = nt * BN;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const long long t0 = tracing ? clock64() : 0;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          if (tracing) t_wait += clock64() - t0;
          uint8_t* sa = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tma_load_2d(sa, &tmA, kb * BK, row0, &full[stage]);
          if (kFused) {
            tma_load_2d(sa + kABytes, &tmB, kb * BK, e * p.N + nt * 128, &full[stage]);
            tma_load_2d(sa + kABytes + kBBytes / 2, &tmB, kb * BK, e * p.N + I + nt * 128,
                        &full[stage]);
          } else {
            tma_load_2d(sa + kABytes, &tmB, kb * BK, e * p.N + n0, &full[stage]);
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (tracing) s_trace[1] = t_wait;
      // let the last loads land before the CTA can exit
      const int outstanding = issued < kStages ? issued : kStages;
      for (int i = 1; i <= outstanding; ++i) {
        int s = stage - i;
        uint32_t ph = phase;
        if (s < 0) { s += kStages; ph ^= 1u; }
        drain(&full[s], ph);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_mx8(BM, BN);
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0, acc_phase = 0;
      unsigned long long t_tmem = 0, t_data = 0, t_sf = 0, nkb = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const long long ta = tracing ? clock64() : 0;
        if (!mbar_wait(tempty, acc_phase ^ 1u, abort_flag, p.status)) break;
        if (tracing) t_tmem += clock64() - ta;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const uint32_t sf_tmem = tmem_base + static_cast<uint32_t>(kSfCol + slot * kSfSlotCols);
          if ((kb & 3) == 0) {
            const long long t0 = tracing ? clock64() : 0;
            if (!mbar_wait(&sf_full[slot], sphase, abort_flag, p.status)) { ok = false; break; }
            if (tracing) t_sf += clock64() - t0;
            tc_fence_after();
            const uint32_t ss = smem_u32(smem + kSfOffset + slot * kSfSlotBytes);
            tc_cp_32x128b_x4(sf_tmem + 0, rows16_desc(ss));
            tc_cp_32x128b_x4(sf_tmem + 4, rows16_desc(ss + kSfBytesA));
            tc_cp_32x128b_x4(sf_tmem + 8, rows16_desc(ss + kSfBytesA + 512));
          }
          const long long t1 = tracing ? clock64() : 0;
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          if (tracing) {
            t_data += clock64() - t1;
            ++nkb;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint32_t id = idesc_with_sf(idesc, kb & 3, kb & 3);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            tc_mma_mx8(tmem_base, sw128_kmajor_desc(sa + k * UMMA_K),
                       sw128_kmajor_desc(sb + k * UMMA_K), id, sf_tmem, sf_tmem + 4,
                       (kb > 0 || k > 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if ((kb & 3) == 3 || kb == KB - 1) {
            tc_commit(&sf_empty[slot]);
            if (++slot == kSfSlots) { slot = 0; sphase ^= 1u; }
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(tfull);
        acc_phase ^= 1u;
      }
      if (tracing) {
        s_trace[2] = t_tmem;
        s_trace[3] = t_data;
        s_trace[4] = t_sf;
        s_trace[7] = nkb;
      }
      // every MMA issued so far must complete before TMEM is released
      tc_commit(mma_done);
      drain(mma_done, 0);
    }
  } else if (warp == 2) {
    // -------------------------------------------------------- scale loader
    int slot = 0;
    uint32_t sphase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int e, row0, rows, nt;
      tile_coords(tile, e, row0, rows, nt);
      // weight-scale blocks of the B tile's two 128-row halves
      const int nbh0 = kFused ? nt : nt * 2;
      const int nbh1 = kFused ? I / 128 + nt : nbh0 + 1;
      bool ok = true;
      for (int g = 0; g < KG; ++g) {
        const bool got = mbar_wait_warp(&sf_empty[slot], sphase ^ 1u, abort_flag, p.status);
        if (!got) { ok = false; break; }
        uint32_t a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t r = static_cast<int64_t>(row0) + lane + 32 * j;
          a[j] = r < p.M_cap ? p.a_scale[static_cast<int64_t>(g) * p.ld_as + r] : 0x7F7F7F7Fu;
        }
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint8_t* ws =
              p.w_scale + (static_cast<int64_t>(e) * NB + (h ? nbh1 : nbh0)) * KB + 4 * g;
          uint32_t word = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            word |= static_cast<uint32_t>(4 * g + b < KB ? ws[b] : 127u) << (8 * b);
          w[h] = word;
        }
        const uint32_t ss = smem_u32(smem + kSfOffset + slot * kSfSlotBytes);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ss + lane * 16), "r"(a[0]),
                     "r"(a[1]), "r"(a[2]), "r"(a[3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(ss + kSfBytesA + lane * 16),
                     "r"(w[0])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(ss + kSfBytesA + 512 +
                                                                       lane * 16),
                     "r"(w[1])
                     : "memory");
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[slot]);
        if (++slot == kSfSlots) { slot = 0; sphase ^= 1u; }
      }
      if (!ok) break;
    }
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kFirstEpiWarp;
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int half = ew >> 2;      // which 128 of the 256 columns
    uint32_t acc_phase = 0;
    unsigned long long t_ewait = 0, t_ework = 0;
    int iter = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++iter) {
      int e, row0, rows, nt;
      tile_coords(tile, e, row0, rows, nt);
      const long long t0 = tracing ? clock64() : 0;
      const int row_in_tile = quarter * 32 + lane;
      const int row = row0 + row_in_tile;
      const bool row_ok = row_in_tile < rows && row < p.M_cap;
      const bool got = mbar_wait_warp(tfull, acc_phase, abort_flag, p.status);
      if (!got) break;
      const long long t1 = tracing ? clock64() : 0;
      tc_fence_after();
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      // stand-alone: columns [128 half, +128); fused: gate [64 half, +64)
      // and up [128 + 64 half, +64)
      const uint32_t c_lo = kFused ? static_cast<uint32_t>(64 * half) : static_cast<uint32_t>(128 * half);
      const uint32_t c_hi = kFused ? static_cast<uint32_t>(128 + 64 * half) : c_lo + 64u;
      uint32_t v0[32], v1[32], v2[32], v3[32];
      tc_ld32(tq + c_lo, v0);
      tc_ld32(tq + c_lo + 32, v1);
      tc_ld32(tq + c_hi, v2);
      tc_ld32(tq + c_hi + 32, v3);
      tc_wait64(v0, v1);
      tc_regs_landed(v2);
      tc_regs_landed(v3);
      // the accumulator is free for the next tile's MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      acc_phase ^= 1u;
      if constexpr (kFused) {
        // h = bf16(silu(bf16 g) * bf16 u), kept in v0/v1; this half's row max
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float h0 = silu_mul_bf16(bf16_round(__uint_as_float(v0[j])),
                                         bf16_round(__uint_as_float(v2[j])));
          const float h1 = silu_mul_bf16(bf16_round(__uint_as_float(v1[j])),
                                         bf16_round(__uint_as_float(v3[j])));
          v0[j] = __float_as_uint(h0);
          v1[j] = __float_as_uint(h1);
          m = fmaxf(m, fmaxf(fabsf(h0), fabsf(h1)));
        }
        // the other half's maximum for the same row (double-buffered by tile)
        const int par = iter & 1;
        s_amax[(par * 2 + half) * 128 + row_in_tile] = m;
        __syncwarp();
        if (lane == 0) mbar_arrive(&amax_bar[quarter]);
        const bool got2 = mbar_wait_warp(&amax_bar[quarter], static_cast<uint32_t>(par),
                                         abort_flag, p.status);
        if (!got2) break;
        const float amax = fmaxf(m, s_amax[(par * 2 + (half ^ 1)) * 128 + row_in_tile]);
        float sc, inv;
        uint32_t b;
        group_scale(amax, true, sc, inv, b);
        if (row_ok) {
          const int t = nt;
          uint4* dst = reinterpret_cast<uint4*>(p.di + static_cast<int64_t>(row) * I + t * 128 +
                                                half * 64);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) h[j] = __uint_as_float(v0[16 * q + j]);
            const uint2 lo = fp8x8(h, inv), hi = fp8x8(h + 8, inv);
            dst[q] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) h[j] = __uint_as_float(v1[16 * q + j]);
            const uint2 lo = fp8x8(h, inv), hi = fp8x8(h + 8, inv);
            dst[2 + q] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
          if (half == 0) {
            // byte t%4 of word (t/4, row); the last group also clears the
            // word's unused bytes
            uint8_t* w = p.di_scale + (static_cast<int64_t>(t >> 2) * p.ld_ds + row) * 4;
            w[t & 3] = static_cast<uint8_t>(b);
            if (t == num_n - 1)
              for (int z = (t & 3) + 1; z < 4; ++z) w[z] = 0;
          }
        }
      } else if (row_ok) {
        const int col0 = nt * BN + half * 128;
        const float wm = p.row_w != nullptr ? p.row_w[row] : 1.0f;
        uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row) * p.N + col0);
        auto put = [&](const uint32_t (&v)[32], int q) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 o;
            o.x = bf16x2_bits(__uint_as_float(v[8 * i + 0]) * wm, __uint_as_float(v[8 * i + 1]) * wm);
            o.y = bf16x2_bits(__uint_as_float(v[8 * i + 2]) * wm, __uint_as_float(v[8 * i + 3]) * wm);
            o.z = bf16x2_bits(__uint_as_float(v[8 * i + 4]) * wm, __uint_as_float(v[8 * i + 5]) * wm);
            o.w = bf16x2_bits(__uint_as_float(v[8 * i + 6]) * wm, __uint_as_float(v[8 * i + 7]) * wm);
            dst[q * 4 + i] = o;
          }
        };
        put(v0, 0);
        put(v1, 1);
        put(v2, 2);
        put(v3, 3);
      }
      if (tracing) {
        const long long t2 = clock64();
        t_ewait += t1 - t0;
        t_ework += t2 - t1;
      }
    }
    if (tracing && ew == 0 && lane == 0) {
      s_trace[5] = t_ewait;
      s_trace[6] = t_ework;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (tracing && threadIdx.x == 0) {
    s_trace[0] = static_cast<unsigned long long>(clock64() - t_kernel0);
    for (int i = 0; i < kTraceWords; ++i) p.trace[blockIdx.x * kTraceWords + i] = s_trace[i];
  }
}

}  // namespace mx
}  // namespace

int launch_grouped_gemm_mx(const MxGemmArgs& a, cudaStream_t s) {
  if (a.E > mx::kMaxE) {
    set_error("moe_grouped_gemm: block-scaled path supports E <= %d", mx::kMaxE);
    return MOE_ERR_INVALID_ARG;
  }
  CUtensorMap ta, tb;
  int rc = make_tmap_k128(&ta, a.A, a.Kd, a.M_cap, a.Kd, mx::BM);
  if (rc != MOE_OK) return rc;
  const bool fused = a.di != nullptr;
  rc = make_tmap_k128(&tb, a.W, a.Kd, static_cast<uint64_t>(a.E) * a.N, a.Kd,
                      fused ? mx::BN / 2 : mx::BN);
  if (rc != MOE_OK) return rc;
  mx::Params p;
  p.a_scale = a.A_scale;
  p.ld_as = a.ld_as;
  p.w_scale = a.W_scale;
  p.start = a.start;
  p.tile_prefix = a.tile_prefix;
  p.d_total = a.d_total;
  p.row_w = a.row_w;
  p.E = a.E;
  p.N = a.N;
  p.Kd = a.Kd;
  p.M_cap = a.M_cap;
  p.out = a.out;
  p.status = a.status;
  p.trace = a.trace;
  p.di = a.di;
  p.di_scale = a.di_scale;
  p.ld_ds = a.ld_ds;
  static bool attr_set[4][64] = {};
  const bool trace = p.trace != nullptr;
  void (*kernel)(CUtensorMap, CUtensorMap, mx::Params) =
      fused ? (trace ? mx::grouped_gemm_mx_kernel<true, true> : mx::grouped_gemm_mx_kernel<false, true>)
            : (trace ? mx::grouped_gemm_mx_kernel<true, false> : mx::grouped_gemm_mx_kernel<false, false>);
  const int variant = (fused ? 2 : 0) + (trace ? 1 : 0);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[variant][dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mx::kSmemBytes) != cudaSuccess)
      return check_launch("cudaFuncSetAttribute(grouped_gemm_mx_kernel)");
    attr_set[variant][dev] = true;
  }
  kernel<<<device_sm_count(), mx::kThreads, mx::kSmemBytes, s>>>(ta, tb, p);
  return check_launch("grouped_gemm_mx_kernel");
}

}  // namespace moe
