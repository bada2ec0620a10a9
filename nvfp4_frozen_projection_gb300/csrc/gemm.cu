// NVFP4 frozen-projection GEMM with the fused LoRA branch, for sm_103a.
//
// "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 7:
//   frozen projections = NVFP4 GEMMs with FP32 accumulation and BF16 output
//   (forward Y = X W^T on the cached forward layout, input gradient dX = dY W on
//   the cached backward layout); LoRA branch = BF16 GEMMs on the reconstructed
//   shared input; Figure 3: both branches sum into the layer output.
//
//   OUT[m, n] = s * ( sum_k A[m,k] B[n,k]  +  sum_j LA[m,j] LB[n,j] )  [+ ADD[m, n]]
//
// A [M, K] and B [N, K] are NVFP4 (E2M1 codes + UE4M3 scales per 16 along K); the
// first sum runs on the block-scaled tensor cores (tcgen05.mma kind::mxf4nvf4,
// block16).  LA [M, RPE] and LB [N, RPE] are BF16: the LoRA down-projection
// output, pre-scaled so that s * LA LB^T equals the LoRA term and stored as a
// hi/lo BF16 pair, and the LoRA up-projection stored twice; their product runs as
// tcgen05.mma kind::f16 (K = 16 per instruction) into the same TMEM accumulator.
// RPE is 32, 64 or 128 columns, loaded in 128-byte (or one 64-byte) swizzled
// chunks.  s = g_a * g_b (or 1 when either per-tensor scale is zero, in which
// case the NVFP4 operand is all zero).
//
// Structure: one persistent CTA per SM, 14 warps.  Tiles 256 wide run on CTA
// pairs (clusters of two along M, .cta_group::2 MMAs over 256 rows); tiles 128
// wide run on single CTAs.  Every CTA loads its own operands: no TMA copy is
// multicast.
//   warp 0      TMA producer: A/B tiles (128-byte rows, 128B swizzle; one 16 KB
//               A box per CTA and, for a pair, half of the B tile each) and
//               the scale-factor atoms (tiled copies: one box of 4 atoms per
//               row block; plain bulk copies measured ~8 % slower) into a STAGES-deep
//               shared-memory ring; the LoRA operands once per tile.
//   warp 1      TMEM allocator and MMA issuer (one thread): MMAs only;
//               tcgen05.commit frees ring slots (in both CTAs of the pair) and
//               publishes the accumulator.
//   warps 2-5   scale staging: shared -> TMEM with tcgen05.st (one warp per TMEM
//               lane quarter).  A tcgen05.cp per atom on the MMA issuer's pipe
//               cost ~35 extra cycles per copy beyond one per MMA; TMEM stores
//               from other warps do not slow the MMAs.
//   warps 6-13  epilogue: TMEM -> registers (tcgen05.ld) 32 columns at a time,
//               each slice scaled, added to the prefetched addend and rounded to
//               BF16 at once, so the single accumulator is released as soon as the
//               last slice has landed; then swizzled staging and TMA stores,
//               optional amax.
// Tiles are visited in bands of M-units swept over all N-tiles (see unit_mn), so
// a large A operand leaves DRAM once.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pact {

#ifndef PACT_DEBUG
__device__ unsigned g_pact_status;
#endif

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
// FP4 elements of K per ring stage: 128-byte tile rows, so each stage moves one
// 16 KB A box and one 32 KB B box (TMA throughput grows with box size; 64-byte
// rows measured slower even with twice the ring depth).
constexpr int kStageK = 256;

// Shared memory: [ring: STAGES x (A | B | SFA | SFB)] [LA] [LB] [epilogue staging]
// [barriers].  A stage's scale factors travel with its A/B tiles (loaded after
// them, on the same barrier): issuing them apart or ahead measured slower.
// PAIR: the tile is computed by a CTA pair with .cta_group::2 MMAs (M = 256 over the
// pair): each CTA holds its 128 A rows and half of the B tile (and of the LoRA
// up-projection rows); the scale factors of all BN B rows are staged in both.
template <int BN, int BK, int STAGES, int RPE, bool PAIR = false>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int ROWB = BK / 2;   // bytes of one tile row per stage
  static constexpr int KSUB = BK / 64;  // K=64 MMAs per stage
  static constexpr int NRB = BN / 128;  // 128-row scale atoms of the B tile
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows in this CTA's shared memory
  static constexpr int A_BYTES = BM * ROWB;
  static constexpr int B_BYTES = B_ROWS * ROWB;
  static constexpr int SFA_BYTES = KSUB * 512;
  static constexpr int SFB_BYTES = NRB * KSUB * 512;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // LoRA operands: LA [BM, RPE] = the down-projection output as a hi|lo BF16 pair,
  // LB [BN, RP] = the up-projection (RP = RPE/2 columns), read by both the hi and the
  // lo MMAs.  Each is loaded in chunks of at most 64 columns (128-byte rows).
  static constexpr int RP = RPE / 2;
  static constexpr int LA_CH = RPE * 2 > 128 ? 128 : RPE * 2;  // row bytes of an LA chunk
  static constexpr int LB_CH = RP * 2 > 128 ? 128 : RP * 2;
  static constexpr int NLA = RPE * 2 / LA_CH;
  static constexpr int NLB = RP * 2 / LB_CH;
  static constexpr int LA_CHUNK = BM * LA_CH;
  static constexpr int LB_CHUNK = B_ROWS * LB_CH;
  static constexpr int LA_OFF = STAGES * STAGE_BYTES;
  static constexpr int LA_BYTES = NLA * LA_CHUNK;
  static constexpr int LB_OFF = LA_OFF + LA_BYTES;
  static constexpr int LB_BYTES = NLB * LB_CHUNK;
  // Epilogue staging for TMA stores: per epilogue warp NSTG buffers of 32 rows x 32
  // BF16 columns (2 KB, 64-byte swizzled rows); double-buffered when shared memory
  // allows.
  static constexpr int STG_OFF = LB_OFF + LB_BYTES;
  static constexpr int STG_BUF = 2048;
  static constexpr int NSTG = (STG_OFF + 2 * 8 * STG_BUF + 512 + 1024 <= 232448) ? 2 : 1;
  static constexpr int BAR_OFF = STG_OFF + NSTG * 8 * STG_BUF;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // + barriers + alignment slack
  static constexpr uint32_t AB_SWZ = ROWB == 128 ? 2u : 4u;  // 128B or 64B swizzle
  static constexpr uint32_t AB_SBO = 8 * ROWB;                // 8-row swizzle atom
  static constexpr uint32_t swz_mode(int row_bytes) {  // 32B -> 6, 64B -> 4, 128B -> 2
    return row_bytes == 32 ? 6u : (row_bytes == 64 ? 4u : 2u);
  }
  static constexpr uint32_t LA_SWZ = swz_mode(LA_CH), LB_SWZ = swz_mode(LB_CH);
  static constexpr uint32_t LA_SBO = 8 * LA_CH, LB_SBO = 8 * LB_CH;  // 8-row swizzle atoms
  static constexpr int LA_STEPS = LA_CH / 32, LB_STEPS = LB_CH / 32;  // K=16 BF16 per step
  static constexpr int SF_BASE = 256;                          // TMEM column
  static constexpr int SF_COLS = 4 * KSUB * (1 + NRB);         // per stage
  static constexpr uint32_t TMEM_COLS = 512;
  // warp 0 TMA, warp 1 MMA, warps 2-5 scale-factor staging, warps 6-13 epilogue
  static constexpr int THREADS = 448;
  static constexpr int SF_WARP0 = 2;
  static constexpr int EPI_WARP0 = 6;
  static constexpr int EPI_THREADS = 256;
  static constexpr int EPI_COLS = BN / 2;    // accumulator columns per epilogue warp
  static constexpr int SFA_TCOLS = 4 * KSUB;        // TMEM columns of a stage's A scales
  static constexpr int SFB_TCOLS = 4 * KSUB * NRB;  // ... and B scales
  // barriers (8 bytes each): full[S], empty[S], sf_full[S] (the stage's scales are
  // in TMEM), then lora_full, lora_empty, acc_full, acc_empty, final, lora_peer
  static constexpr int NBARS = 3 * STAGES + 6;
  static_assert((SFA_TCOLS == 8 || SFA_TCOLS == 16) &&
                    (SFB_TCOLS == 8 || SFB_TCOLS == 16 || SFB_TCOLS == 32),
                "SF staging shapes");
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(BK == 128 || BK == 256, "BK");
  static_assert(RPE == 32 || RPE == 64 || RPE == 128, "RPE");
  static_assert(SF_BASE + STAGES * SF_COLS <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && LA_OFF % 1024 == 0 && LB_OFF % 1024 == 0 &&
                    STG_OFF % 1024 == 0,
                "align");
  static_assert(NBARS * 8 <= 504, "barrier area");
};

// Instruction descriptors (M = 128, or 256 for a CTA pair; K-major A and B, dense).
__host__ __device__ constexpr uint32_t idesc_nvf4(int n, int m = 128) {
  // atype = btype = E2M1 (1), scale type UE4M3 (bit 23 = 0)
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int n, int m = 128) {
  // D = F32 (bits 4-5 = 1), A = B = BF16 (1)
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

// Word i (runtime, 0..15) of sixteen register values, by a chain of selects.
__device__ __forceinline__ uint32_t pick16(const uint32_t* w, int i) {
  uint32_t v = w[15];
#pragma unroll
  for (int k = 14; k >= 0; --k) v = (i == k) ? w[k] : v;
  return v;
}

// silu_mul, kept out of the epilogue's instruction stream (it runs for a few elements
// per warp only).
static __device__ __noinline__ float silu_mul_out_of_line(float g, float u) {
  return silu_mul(g, u);
}

// max(|a|, |b|) of two BF16 pairs, lane by lane (the sign bits are the xor of the
// inputs' and are masked by the caller; a NaN loses to the other operand).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Element e (0..31) of a 32-column BF16 slice held as 16 packed pairs.
__device__ __forceinline__ float slice_elem(const uint32_t (&w)[16], int e) {
  const uint32_t v = pick16(w, e >> 1);
  return __uint_as_float((e & 1) ? (v & 0xFFFF0000u) : (v << 16));
}

// Statistics of the fused gate|up output for the SiLU-multiply quantisation, over
// one lane's row of the tile: the epilogue holds its BF16 results in 32-column
// slices, and in the interleaved order slice 2j is gate and slice 2j + 1 the up of
// the same columns.  ag, au: max |gate|, max |up| (FP32 bits of BF16 values, exact).
// xh: the exact max |h| of this lane's elements so far, h = silu_mul(gate, up) by the
// exact FP32 recipe; xw: the warp's, a lower bound of the tensor's.  The recipe's
// s = RN(g / RN(1 + e)) satisfies |s| <= max(g, 0) + 0.28: for g >= 0, RN(1 + e) >= 1
// gives |s| <= g; for g < 0, |g| / (1 + e^-g) <= 0.2785 and the recipe's roundings
// move it by a few units in the last place.  So |h| = |RN(s u)| <=
// RN(RN(max(g, 0) + 0.3) |u|) (rounding is monotonic), and over a slice <=
// RN((max |g| + 0.3) max |u|): a slice where that is below xw holds nothing above it
// (three instructions per slice).  Otherwise the slice's largest per-element bound,
// formed with BF16 roundings (a packed max, add and multiply per two elements),
// decides; only if that reaches xw are the elements whose own FP32 bound reaches xw
// evaluated exactly.  While xw < 2^-100 (the warp's first slices, or tiny values)
// the packed stage is skipped and the lane seeds its threshold with the exact value
// of its element of largest bound.
__device__ __forceinline__ float gu_bound(float g, float u) {
  return __fmul_rn(__fadd_rn(fmaxf(g, 0.0f), 0.3f), fabsf(u));
}

__device__ __forceinline__ void gate_up_slice(const uint32_t (&gs)[16], const uint32_t (&us)[16],
                                              float xw, float& xh, uint32_t& ag, uint32_t& au) {
  uint32_t gm = 0, um = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    gm = bf16x2_max_abs(gm, gs[i]);
    um = bf16x2_max_abs(um, us[i]);
  }
  gm &= 0x7FFF7FFFu;
  um &= 0x7FFF7FFFu;
  const uint32_t gmb = max(gm & 0xFFFFu, gm >> 16) << 16;
  const uint32_t umb = max(um & 0xFFFFu, um >> 16) << 16;
  ag = max(ag, gmb);
  au = max(au, umb);
  const bool all = !(xw >= 0x1p-100f);
  if (!all) {
    if (__fmul_rn(__fadd_rn(__uint_as_float(gmb), 0.3f), __uint_as_float(umb)) < xw) return;
    // the per-element bound with BF16 roundings: v = RN(max(g, 0) + 0.3) >= |s| exactly
    // (g is a BF16 value) and RN_bf16(v |u|) (1 + 2^-8) >= RN(v |u|) >= |h|
    const __nv_bfloat162 zero2 = __float2bfloat162_rn(0.0f), c2 = __float2bfloat162_rn(0.3f);
    uint32_t bm = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t g2 = gs[i], u2 = us[i] & 0x7FFF7FFFu;
      const __nv_bfloat162 v =
          __hadd2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&g2), zero2), c2);
      __nv_bfloat162 bnd = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&u2));
      bm = __vmaxu2(bm, *reinterpret_cast<uint32_t*>(&bnd) & 0x7FFF7FFFu);
    }
    const float bmax = __uint_as_float(max(bm & 0xFFFFu, bm >> 16) << 16);
    if (__fmul_rn(bmax, 1.0f + 0x1p-6f) < xw) return;
  }
  float thr = xw;
  if (all) {
    float best = -1.0f;
    int be = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const uint32_t gv = gs[e >> 1], uv = us[e >> 1];
      const float bnd = gu_bound(__uint_as_float((e & 1) ? (gv & 0xFFFF0000u) : (gv << 16)),
                                 __uint_as_float((e & 1) ? (uv & 0xFFFF0000u) : (uv << 16)));
      if (bnd > best) {
        best = bnd;
        be = e;
      }
    }
    xh = fmaxf(xh, fabsf(silu_mul_out_of_line(slice_elem(gs, be), slice_elem(us, be))));
    thr = fmaxf(xw, xh);
  }
  uint32_t cand = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t gv = gs[e >> 1], uv = us[e >> 1];
    const float bnd = gu_bound(__uint_as_float((e & 1) ? (gv & 0xFFFF0000u) : (gv << 16)),
                               __uint_as_float((e & 1) ? (uv & 0xFFFF0000u) : (uv << 16)));
    cand |= (bnd < thr ? 0u : 1u) << e;
  }
#pragma unroll 1
  while (cand) {
    const int e = __ffs(cand) - 1;
    cand &= cand - 1;
    // a NaN is ignored, as the amax of the oracle ignores it
    xh = fmaxf(xh, fabsf(silu_mul_out_of_line(slice_elem(gs, e), slice_elem(us, e))));
  }
}

// Called by every lane of the warp (live: the lane's row lies inside M); the warp's
// threshold xw is refreshed after each slice pair.
template <int NCH>
__device__ __forceinline__ void gate_up_stats(const uint32_t (&out)[NCH][16], int nbase, int N,
                                              bool live, float& xw, float& xh, uint32_t& ag,
                                              uint32_t& au) {
#pragma unroll
  for (int ch = 0; ch + 1 < NCH; ch += 2) {
    if (nbase + 32 * ch >= N) break;  // the whole slice pair lies past N (uniform)
    if (live) gate_up_slice(out[ch], out[ch + 1], xw, xh, ag, au);
    xw = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(xh)));
  }
}

__device__ __forceinline__ void raise_error(volatile uint32_t* abort_flag, unsigned* status,
                                            unsigned code) {
  *abort_flag = 1u;
  atomicOr(status, code);
}

// CM = CTAs per cluster along M: 1, or 2 for a pair.
// PAIR (CM = 2): the two CTAs of a cluster compute the tiles (m, n) and (m + 1, n)
// as one M = 256 pair MMA issued by the even CTA ("leader"): each CTA loads its A
// tile and half of the B tile (no multicast), stages its scale factors into its own
// TMEM and reports to the leader's barriers (sf_full, acc_empty, lora_peer); the
// leader's commits reach both CTAs.
// GU: the fused gate|up forward (interleaved columns stored back in the logical
// order, amax3 statistics); instantiated only for that call, so the other GEMMs carry
// none of its code.
template <int BN, int BK, int STAGES, int RPE, int CM, bool PAIR = false, bool GU = false>
__global__ void __launch_bounds__(448, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmLA,
                 const __grid_constant__ CUtensorMap tmLB,
                 const __grid_constant__ CUtensorMap tmOut,
                 const __grid_constant__ CUtensorMap tmSFA,
                 const __grid_constant__ CUtensorMap tmSFB, const GemmParams p) {
  static_assert(PAIR ? CM == 2 : CM == 1, "a pair is a cluster of two; other tiles one CTA");
  using C = GemmCfg<BN, BK, STAGES, RPE, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar0 = base + C::BAR_OFF;
  const uint32_t full0 = bar0, empty0 = bar0 + 8 * STAGES;
  const uint32_t sf_full0 = bar0 + 8 * (2 * STAGES);
  const uint32_t lora_full = sf_full0 + 8 * STAGES;
  const uint32_t lora_empty = lora_full + 8;
  const uint32_t acc_full = lora_full + 16;
  const uint32_t acc_empty = lora_full + 24;
  const uint32_t final_bar = lora_full + 32;
  const uint32_t lora_peer = lora_full + 40;  // PAIR: the peer's LoRA operands landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 504);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::BAR_OFF + 508);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nks = (p.K + BK - 1) / BK;
  // work units: CM vertically adjacent tiles (an M-unit) sharing one B tile.  The
  // units are ordered in bands of band_mc M-units: a band is swept over every
  // N-tile, M-units fastest, before the next band starts.  With one band (the
  // whole M range) consecutive units share a B tile and all of A stays in L2
  // across the sweeps; when A is too large for that, a narrower band keeps its
  // rows in L2 while every B tile passes, so each byte of A leaves DRAM once.
  const uint32_t crank = CM > 1 ? cluster_ctarank() : 0u;
  const int num_mc = (p.num_m + CM - 1) / CM;
  const int nunits = num_mc * p.num_n;
  const int unit0 = (int)blockIdx.x / CM, nclusters = (int)gridDim.x / CM;
  const int band = p.band_mc;
  auto unit_mn = [&](int u, int& mc, int& n) {
    const int bi = u / (band * p.num_n), r = u - bi * band * p.num_n;
    const int mc0 = bi * band, bm = min(band, num_mc - mc0);
    n = r / bm;
    mc = mc0 + (r - n * bm);
  };
  auto tile_mt = [&](int u) {
    int mc, n;
    unit_mn(u, mc, n);
    return mc * CM + (int)crank;
  };
  auto tile_n0 = [&](int u) {
    int mc, n;
    unit_mn(u, mc, n);
    return n * BN;
  };
  // this CTA's K steps over all its units, as one sequence of "fills"
  const int my_units = unit0 < nunits ? (nunits - unit0 + nclusters - 1) / nclusters : 0;
  const int nfills = my_units * nks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      // one commit: this CTA's own, or for a pair the leader's (reaching both)
      mbar_init(empty0 + 8 * s, 1);
      // PAIR: one arrival per scale-staging warp of both CTAs (at the leader)
      mbar_init(sf_full0 + 8 * s, PAIR ? 8 : 128);
    }
    mbar_init(lora_full, 1);
    mbar_init(lora_empty, 1);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, PAIR ? 16 : C::EPI_THREADS);  // PAIR: one per epilogue warp, both CTAs
    mbar_init(final_bar, 1);
    mbar_init(lora_peer, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmOut);
    prefetch_tensormap(&tmSFA);
    prefetch_tensormap(&tmSFB);
    if (p.lora_steps) {
      prefetch_tensormap(&tmLA);
      prefetch_tensormap(&tmLB);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CM > 1) cluster_sync();  // peers' barriers are initialised
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // Everything per tile is computed once per tile: the per-stage path between
      // an empty barrier completing and the next copies being issued stays short.
      uint32_t pend = 0, pend_par = 0, lpend = 0, lpend_par = 0;
      uint32_t lphase = 0, phase = 0;
      int stage = 0;
      bool ok = true;
      for (int u = unit0; u < nunits && ok; u += nclusters) {
        const int mt = tile_mt(u);
        const int m0 = mt * C::BM;
        const int n0 = tile_n0(u);
        if (p.lora_steps) {
          if (!mbar_wait(lora_empty, lphase ^ 1u, kWaitLimitNs, abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(lora_full, C::LA_BYTES + C::LB_BYTES);
#pragma unroll
          for (int c = 0; c < C::NLA; ++c)
            tma_load_2d(base + C::LA_OFF + c * C::LA_CHUNK, &tmLA, 64 * c, m0, lora_full);
#pragma unroll
          for (int c = 0; c < C::NLB; ++c)
            tma_load_2d(base + C::LB_OFF + c * C::LB_CHUNK, &tmLB, 64 * c,
                        PAIR ? n0 + (int)crank * C::B_ROWS : n0, lora_full);
          lpend = 1u;
          lpend_par = lphase;
          lphase ^= 1u;
        }
        // a CTA whose m-tile lies past M (odd tile count) computes on zero-filled A
        // and stores nothing; its scale reads stay inside the last row block
        const int sfa_row = min(mt, p.num_m - 1);
        const int nb = n0 + (int)crank * C::B_ROWS;  // this CTA's B rows
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, kWaitLimitNs, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sb = base + stage * C::STAGE_BYTES;
          // tiled copies always deliver whole boxes (zero fill past K and past N)
          mbar_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(sb, &tmA, ks * C::ROWB, m0, fb);
          tma_load_2d(sb + C::A_BYTES, &tmB, ks * C::ROWB, nb, fb);
          // the stage's scale atoms: 4 of the A row block, 4 of each B row block
          // (x in 8-byte elements: 64 per atom)
          tma_load_2d(sb + C::A_BYTES + C::B_BYTES, &tmSFA, ks * C::KSUB * 64, sfa_row, fb);
          tma_load_2d(sb + C::A_BYTES + C::B_BYTES + C::SFA_BYTES, &tmSFB, ks * C::KSUB * 64,
                      n0 / 128, fb);
          pend |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        raise_error(abort_flag, p.status, PACT_DEV_TIMEOUT | PACT_DEV_ROLE_TMA);
        // let copies already in flight land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if (pend & (1u << s)) mbar_wait(full0 + 8 * s, (pend_par >> s) & 1u, 10000000ull, nullptr);
        if (lpend) mbar_wait(lora_full, lpend_par, 10000000ull, nullptr);
      } else if constexpr (CM > 1) {
        // the peer's MMA commits arrive on this CTA's empty barriers: wait for the
        // release of the last STAGES loads before the CTA may exit
        for (int i = 0; i < STAGES; ++i) {
          mbar_wait(empty0 + 8 * stage, phase ^ 1u, kWaitLimitNs, abort_flag);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (PAIR && crank != 0) {
      // the peer: tell the leader when this CTA's LoRA operands have landed
      if (lane == 0 && p.lora_steps) {
        uint32_t lphase = 0;
        for (int u = unit0; u < nunits; u += nclusters) {
          if (!mbar_wait(lora_full, lphase, kWaitLimitNs, abort_flag)) {
            raise_error(abort_flag, p.status, PACT_DEV_TIMEOUT | PACT_DEV_ROLE_MMA);
            break;
          }
          mbar_arrive_cta(lora_peer, 0);
          lphase ^= 1u;
        }
      }
    } else if (lane == 0) {
      uint32_t lphase = 0, aphase = 0, phase = 0;
      int stage = 0;
      bool ok = true;
      constexpr int MM = PAIR ? 256 : 128;
      const uint32_t idesc = idesc_nvf4(BN, MM);
      const uint32_t idesc_l = idesc_bf16(BN, MM);
      auto wait_x = [&](uint32_t bar, uint32_t par) {  // barriers the peer also arrives on
        return PAIR ? mbar_wait_cluster(bar, par, kWaitLimitNs, abort_flag)
                    : mbar_wait(bar, par, kWaitLimitNs, abort_flag);
      };
      // descriptors of stage 0 (a stage's are these plus its offset in 16-byte units:
      // every operand address stays inside the 14-bit start-address field)
      const uint64_t da0 = smem_desc(base, 16, C::AB_SBO, C::AB_SWZ);
      const uint64_t db0 = smem_desc(base + C::A_BYTES, 16, C::AB_SBO, C::AB_SWZ);
      const uint32_t tsf0 = tmem + C::SF_BASE;
      const int nks_full = p.K / BK;
      auto issue_nvf4 = [&](uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb, uint32_t acc) {
        if constexpr (PAIR)
          mma_nvf4_pair(tmem, a, b, idesc, sfa, sfb, acc);
        else
          mma_nvf4(tmem, a, b, idesc, sfa, sfb, acc);
      };
      auto commit_all = [&](uint32_t bar) {  // reaches both CTAs of a cluster
        if constexpr (PAIR)
          mma_commit_pair(bar, (uint16_t)3u);
        else
          mma_commit(bar);
      };
      for (int u = unit0; u < nunits && ok; u += nclusters) {
        if (!wait_x(acc_empty, aphase ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t accum = 0;
        if (p.lora_steps) {
          if (!mbar_wait(lora_full, lphase, kWaitLimitNs, abort_flag) ||
              (PAIR && !wait_x(lora_peer, lphase))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int j = 0; j < p.lora_steps; ++j) {
            // step j reads columns [16j, 16j+16) of LA (hi then lo) and the same
            // up-projection columns [16(j mod RP/16), ...) of LB for both halves
            const int jb = j % (C::RP / 16);
            const uint64_t da = smem_desc(base + C::LA_OFF + (j / C::LA_STEPS) * C::LA_CHUNK +
                                              32u * (uint32_t)(j % C::LA_STEPS),
                                          16, C::LA_SBO, C::LA_SWZ);
            const uint64_t db = smem_desc(base + C::LB_OFF + (jb / C::LB_STEPS) * C::LB_CHUNK +
                                              32u * (uint32_t)(jb % C::LB_STEPS),
                                          16, C::LB_SBO, C::LB_SWZ);
            if constexpr (PAIR)
              mma_bf16_pair(tmem, da, db, idesc_l, accum);
            else
              mma_bf16(tmem, da, db, idesc_l, accum);
            accum = 1;
          }
          if constexpr (PAIR)
            commit_all(lora_empty);
          else
            mma_commit(lora_empty);
          lphase ^= 1u;
        }
        for (int ks = 0; ks < nks; ++ks) {
          // the stage's A/B tiles are in shared memory and its scales in TMEM (for a
          // pair: in both CTAs)
          if (!wait_x(sf_full0 + 8 * stage, phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // this thread's instruction latency between MMAs is what the tensor pipe
          // sees, so a whole stage is issued unrolled from precomputed descriptors
          // (the runtime-count loop measured 15-18 % slower per stage)
          const uint64_t soff = (uint64_t)(stage * (C::STAGE_BYTES >> 4));
          const uint64_t da = da0 + soff, db = db0 + soff;
          const uint32_t tsf = tsf0 + (uint32_t)(stage * C::SF_COLS);
          if (ks < nks_full) {
#pragma unroll
            for (int j = 0; j < C::KSUB; ++j)
              issue_nvf4(da + 2u * j, db + 2u * j, tsf + 4 * j, tsf + 4 * C::KSUB + j * C::NRB * 4,
                         j == 0 ? accum : 1u);
          } else {  // K tail: ksub < KSUB 64-wide steps
            const int ksub = (p.K - ks * BK) / 64;
            for (int j = 0; j < ksub; ++j)
              issue_nvf4(da + 2u * j, db + 2u * j, tsf + 4 * j, tsf + 4 * C::KSUB + j * C::NRB * 4,
                         j == 0 ? accum : 1u);
          }
          accum = 1;
          commit_all(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          commit_all(acc_full);
        else
          mma_commit(acc_full);
        aphase ^= 1u;
      }
      if (!ok) raise_error(abort_flag, p.status, PACT_DEV_TIMEOUT | PACT_DEV_ROLE_MMA);
      // every MMA issued by this thread has completed once final_bar flips
      if constexpr (PAIR)
        mma_commit_pair(final_bar, (uint16_t)1u);
      else
        mma_commit(final_bar);
      mbar_wait(final_bar, 0, kWaitLimitNs, nullptr);
    }
  } else if (warp >= C::SF_WARP0 && warp < C::SF_WARP0 + 4) {
    // ------------------------------------------------------------ scale staging
    // One warp per TMEM lane quarter q.  A 512-byte scale atom holds rows r, r+32,
    // r+64, r+96 in its 16-byte row r (4 bytes = 4 blocks each).  The MMA reads the
    // A scales of tile row 32q + r from TMEM lane 32q + r, column q of the atom's 4
    // columns, and the B scales of every row from lane 32q + (row mod 32) of the
    // lane quarter it computes in, all 4 columns (the atom image itself, in every
    // quarter).  So lane r of warp q loads only 4 bytes of every A atom (columns
    // nobody reads get copies) and the 16-byte rows of the B atoms: 18 KB of
    // shared-memory reads per stage instead of 24 KB, which matters because
    // shared-memory bandwidth is what this pipeline is short of.  Plain TMEM stores
    // keep the MMA issuer's tensor pipe for MMAs only.  The stage's TMEM slot is
    // free again once its full barrier completes: the producer only refills a stage
    // after the MMAs that read it have completed.
    const uint32_t q = (uint32_t)(warp & 3);
    bool ok = true;
    int stage = 0;
    uint32_t phase = 0;
    for (int f = 0; f < nfills; ++f) {
      if (!mbar_wait(full0 + 8 * stage, phase, kWaitLimitNs, abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* sf_p = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES + 16 * lane;
      uint32_t va[C::SFA_TCOLS], vb[C::SFB_TCOLS];
#pragma unroll
      for (int j = 0; j < C::KSUB; ++j) {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(sf_p + 512 * j + 4 * q);
#pragma unroll
        for (int i = 0; i < 4; ++i) va[4 * j + i] = a;
#pragma unroll
        for (int rb = 0; rb < C::NRB; ++rb) {
          const int c = 4 * (j * C::NRB + rb);
          const uint4 b =
              *reinterpret_cast<const uint4*>(sf_p + C::SFA_BYTES + rb * C::KSUB * 512 + 512 * j);
          vb[c] = b.x;
          vb[c + 1] = b.y;
          vb[c + 2] = b.z;
          vb[c + 3] = b.w;
        }
      }
      tc_fence_after();
      const uint32_t tsf = tmem + (q * 32u << 16) + C::SF_BASE + stage * C::SF_COLS;
      tmem_st<C::SFA_TCOLS>(tsf, va);
      tmem_st<C::SFB_TCOLS>(tsf + C::SFA_TCOLS, vb);
      tmem_st_wait();
      tc_fence_before();
      if constexpr (PAIR) {
        // one arrival per warp, at the leader (which issues the pair MMAs)
        __syncwarp();
        if (lane == 0) mbar_arrive_cta_relaxed(sf_full0 + 8 * stage, 0u);
      } else {
        mbar_arrive(sf_full0 + 8 * stage);
      }
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) raise_error(abort_flag, p.status, PACT_DEV_TIMEOUT | PACT_DEV_ROLE_SF);
  } else if (warp >= C::EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    // Two warps per TMEM lane quarter, each owning half of the tile's columns.  The
    // MMA issuer has one accumulator, so the next tile's mainloop waits for this
    // drain: a warp loads its share 32 columns at a time and turns each slice into
    // rounded BF16 (scaled, plus the addend; packed FP32 pairs) at once, so the
    // whole share fits in registers, and the accumulator is released as soon as the
    // last slice has landed, before that slice is converted (measured on GB300: the
    // step's GEMMs 1-4 % faster than a release after the last conversion).  The
    // addend share is fetched, as BF16, while the mainloop still runs.  Then each
    // 32x32 BF16 block (row per lane) goes to a shared staging buffer and out with
    // one TMA store, which also clips rows >= M; rows past M never read addend.
    constexpr int NCH = C::EPI_COLS / 32;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - C::EPI_WARP0;
    const int c0 = (ew >> 2) * C::EPI_COLS;
    const uint32_t stg = base + C::STG_OFF + (uint32_t)(ew * C::NSTG * C::STG_BUF);
    const float ga = *p.ga, gb = *p.gb;
    const float s_main = (ga > 0.0f && gb > 0.0f) ? __fmul_rn(ga, gb) : 1.0f;
    uint32_t amax = 0;  // packed BF16 pairs while the tiles are drained, FP32 bits after
    const bool want_amax = p.out_amax != nullptr;
    uint32_t aphase = 0;
    uint32_t nstore = 0;
    float gu_xh = 0.0f, gu_xw = 0.0f;  // gate|up statistics (amax3): lane's and warp's
    uint32_t gu_ag = 0, gu_au = 0;
    for (int u = unit0; u < nunits; u += nclusters) {
      const int m0 = tile_mt(u) * C::BM;
      const int n0 = tile_n0(u);
      const int m = m0 + q * 32 + lane;
      const bool row_ok = m < p.M;
      // the 32-row block is wholly past M (ragged or padding tile): nothing to store
      const bool blk_live = m0 + q * 32 < p.M;
      // out[ch] first holds the addend slice ch (packed BF16), then the result
      uint32_t out[NCH][16];
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int n = n0 + c0 + 32 * ch;
        if (p.addend && row_ok && n < p.N) {
          const uint16_t* ap = p.addend + (size_t)m * p.N + n;
          if (p.addend32) {
            // a lane reads its own row: 32-byte loads fill whole sectors, so each
            // load instruction costs half the L1 transactions of 16-byte ones (the
            // MIO queue these share with the scale-staging warps' shared loads), and
            // they do not allocate in L1, which the ring leaves small and which
            // nothing reads twice (the o and down forwards 6-7 % faster on GB300)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint32_t* o8 = &out[ch][8 * k];
              asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                           : "=r"(o8[0]), "=r"(o8[1]), "=r"(o8[2]), "=r"(o8[3]), "=r"(o8[4]),
                             "=r"(o8[5]), "=r"(o8[6]), "=r"(o8[7])
                           : "l"(ap + 16 * k));
            }
          } else {
            const uint4* ad = reinterpret_cast<const uint4*>(ap);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 a4 = ad[k];
              out[ch][4 * k] = a4.x;
              out[ch][4 * k + 1] = a4.y;
              out[ch][4 * k + 2] = a4.z;
              out[ch][4 * k + 3] = a4.w;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) out[ch][i] = 0u;
        }
      }
      if (!(PAIR ? mbar_wait_cluster(acc_full, aphase, kWaitLimitNs, abort_flag)
                 : mbar_wait(acc_full, aphase, kWaitLimitNs, abort_flag))) {
        raise_error(abort_flag, p.status, PACT_DEV_TIMEOUT | PACT_DEV_ROLE_EPI);
        break;
      }
      tc_fence_after();
      auto release_acc = [&]() {
        tc_fence_before();
        if constexpr (PAIR) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cta_relaxed(acc_empty, 0u);  // at the leader
        } else {
          mbar_arrive(acc_empty);
        }
      };
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t v[32];
        tmem_ld32(tq + 32u * ch, v);
        tmem_ld_wait();
        // the accumulator is released as soon as the last slice has landed in
        // registers, before that slice is converted
        if (ch == NCH - 1) release_acc();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // packed FP32 pairs: each lane rounds as the scalar operation does
          float2 f = __fmul2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                make_float2(s_main, s_main));
          if (p.addend)  // an absent addend slice is zeros: x + 0 = x for x != -0
            f = __fadd2_rn(f, make_float2(__uint_as_float(out[ch][i] << 16),
                                          __uint_as_float(out[ch][i] & 0xFFFF0000u)));
          out[ch][i] = pack_bf16x2(f.x, f.y);
        }
      }
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int n = n0 + c0 + 32 * ch;
        if (n >= p.N || !blk_live) continue;  // uniform across the warp (N % 32 == 0)
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) PACT_NAN_BF16X2(out[ch][i]);
        }
        if (want_amax && row_ok) {  // packed max |.| of BF16 pairs (signs masked at the end)
#pragma unroll
          for (int i = 0; i < 16; ++i)
            asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(amax) : "r"(amax), "r"(out[ch][i]));
        }
        // staging buffer nstore % NSTG: wait until its previous store has read it
        const uint32_t buf = stg + (nstore % C::NSTG) * C::STG_BUF;
        if (nstore >= (uint32_t)C::NSTG && lane == 0) bulk_wait_read<C::NSTG - 1>();
        __syncwarp();
        // 64-byte swizzle (the store's tensor map says the same): 16-byte chunk k
        // of row r sits at chunk k ^ ((r / 2) % 4), which spreads a store
        // instruction's 32 rows over all banks
        uint8_t* row = smem + (buf - base) + 64 * lane;
        const uint32_t sw = (uint32_t)(lane >> 1) & 3u;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(row + 16 * (k ^ sw)) =
              make_uint4(out[ch][4 * k], out[ch][4 * k + 1], out[ch][4 * k + 2], out[ch][4 * k + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // the interleaved gate|up order goes back to the logical columns here
          tma_store_2d(&tmOut, buf, GU ? (int)gu_logical(n, p.gu_half) : n, m0 + q * 32);
          bulk_commit();
        }
        ++nstore;
      }
      if constexpr (GU) gate_up_stats<NCH>(out, n0 + c0, p.N, row_ok, gu_xw, gu_xh, gu_ag, gu_au);
      aphase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();
    if (want_amax) {
      amax &= 0x7FFF7FFFu;
      amax = __reduce_max_sync(0xFFFFFFFFu, max(amax << 16, amax & 0xFFFF0000u));
      if (lane == 0 && amax) atomicMax(p.out_amax, amax);
    }
    if constexpr (GU) {  // order: h, gate, up
      const uint32_t hx = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(gu_xh));
      const uint32_t gx = __reduce_max_sync(0xFFFFFFFFu, gu_ag);
      const uint32_t ux = __reduce_max_sync(0xFFFFFFFFu, gu_au);
      if (lane == 0) {
        if (hx) atomicMax(p.amax3, hx);
        if (gx) atomicMax(p.amax3 + 1, gx);
        if (ux) atomicMax(p.amax3 + 2, ux);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if constexpr (CM > 1) cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else
      tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
template <int BN, int BK, int STAGES, int RPE, int CM, bool PAIR = false, bool GU = false>
static cudaError_t launch_cfg(const GemmLaunch& L, cudaStream_t stream) {
  using C = GemmCfg<BN, BK, STAGES, RPE, PAIR>;
  auto kern = k_gemm_nvfp4<BN, BK, STAGES, RPE, CM, PAIR, GU>;
  // per device: shared-memory attribute set, and how many clusters fit at once
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CM;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int n = L.num_sms / CM;
    if (CM > 1) {
      cfg.gridDim = dim3(L.num_sms / CM * CM);
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
    }
    max_clusters[dev] = n;
  }
  const int num_mc = (L.p.num_m + CM - 1) / CM;
  const int units = num_mc * L.p.num_n;
  const int clusters = units < max_clusters[dev] ? units : max_clusters[dev];
  cfg.gridDim = dim3(clusters * CM);
  // one band while A (the codes of all M rows) fits comfortably in L2 next to the
  // B tiles in flight; else bands just wide enough to keep every cluster busy
  GemmParams p = L.p;
  const double a_bytes = (double)p.num_m * 128.0 * (double)p.K * 0.5625;
  p.band_mc = num_mc;
  if (a_bytes > 32.0 * 1024 * 1024) {
    const int b = (clusters + p.num_n - 1) / p.num_n;
    p.band_mc = b < 1 ? 1 : (b > num_mc ? num_mc : b);
  }
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, L.tmA, L.tmB, L.tmLA, L.tmLB, L.tmOut, L.tmSFA, L.tmSFB,
                            p);
}

int gemm_block_n(int64_t N, int rpe) { return (N % 256 == 0 && rpe <= 64) ? 256 : 128; }

int gemm_stage_row_bytes() { return kStageK / 2; }

bool gemm_uses_pair(int64_t M, int64_t N, int rpe) {
  return M > 128 && gemm_block_n(N, rpe) == 256;
}

int gemm_cluster_m(int64_t M, int64_t N, int rpe) { return gemm_uses_pair(M, N, rpe) ? 2 : 1; }

// Ring depth: as many stages as shared memory holds next to the LoRA operands and
// one staging buffer per epilogue warp, within the TMEM left for scale factors, at
// most 10.
template <int BN, int BK, int RPE, bool PAIR = false>
constexpr int ring_stages() {
  constexpr int brows = PAIR ? BN / 2 : BN;  // B rows held by one CTA
  constexpr int stage = 128 * BK / 2 + brows * BK / 2 + (BK / 64) * 512 * (1 + BN / 128);
  constexpr int fixed = 128 * RPE * 2 + brows * (RPE / 2) * 2 + 8 * 2048 + 1536;
  constexpr int by_smem = (232448 - fixed) / stage;
  constexpr int by_tmem = 256 / (4 * (BK / 64) * (1 + BN / 128));
  constexpr int s = by_smem < by_tmem ? by_smem : by_tmem;
  return s < 10 ? s : 10;
}

template <int BN, int RPE, int CM, bool GU>
static cudaError_t launch_one(const GemmLaunch& L, cudaStream_t stream) {
  return launch_cfg<BN, kStageK, ring_stages<BN, kStageK, RPE>(), RPE, CM, false, GU>(L, stream);
}

template <int BN, int RPE, bool GU>
static cudaError_t launch_pair(const GemmLaunch& L, cudaStream_t stream) {
  return launch_cfg<BN, kStageK, ring_stages<BN, kStageK, RPE, true>(), RPE, 2, true, GU>(L,
                                                                                       stream);
}

template <bool GU>
static cudaError_t launch_gemm_gu(const GemmLaunch& L, int bn, int rpe, int cm,
                                  cudaStream_t stream) {
  if (bn == 256) {
    if (cm == 2) {
      if (rpe == 32) return launch_pair<256, 32, GU>(L, stream);
      return launch_pair<256, 64, GU>(L, stream);
    }
    if (rpe == 32) return launch_one<256, 32, 1, GU>(L, stream);
    return launch_one<256, 64, 1, GU>(L, stream);
  }
  if (rpe == 32) return launch_one<128, 32, 1, GU>(L, stream);
  if (rpe == 64) return launch_one<128, 64, 1, GU>(L, stream);
  return launch_one<128, 128, 1, GU>(L, stream);
}

cudaError_t launch_gemm_nvfp4(const GemmLaunch& L, int bn, int rpe, int cm, cudaStream_t stream) {
  return L.p.gu_half ? launch_gemm_gu<true>(L, bn, rpe, cm, stream)
                     : launch_gemm_gu<false>(L, bn, rpe, cm, stream);
}

// Test of the bounded-wait path: one thread waits on an mbarrier that nothing
// arrives at, with the same wait routine the GEMM uses and a limit of limit_ns.
// When it gives up it records the timeout in the status word and returns, so the
// context stays usable.
__global__ void k_wait_timeout(uint64_t limit_ns, unsigned* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t never;
  if (threadIdx.x == 0) {
    never = 0u;
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait(smem_addr(&bar), 0, limit_ns, &never)) atomicOr(status, PACT_DEV_TIMEOUT);
  }
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  unsigned* status = nullptr;
  cudaError_t e = status_word_ptr(&status);
  if (e != cudaSuccess) return e;
  note_launch();
  k_wait_timeout<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

// Evaluates one bounds check that fails (index n of an n-element range) without
// touching memory: the debug build records PACT_DEV_BOUNDS, the release build
// compiles the check to true and records nothing.
__global__ void k_bounds_check(int n, int* sink) {
  const int i = n;
  if (!PACT_IN(i < n)) return;
  if (sink) sink[0] = i;  // never reached with sink null (the launch passes null)
}

cudaError_t launch_bounds_check(cudaStream_t stream) {
  note_launch();
  k_bounds_check<<<1, 1, 0, stream>>>(1, nullptr);
  return cudaGetLastError();
}

cudaError_t status_word_ptr(unsigned** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_pact_status);
}

}  // namespace pact
