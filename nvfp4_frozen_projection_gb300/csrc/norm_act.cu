// Fused nonlinear kernels around the NVFP4 projections.
//
// "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 7:
//   RMSNorm        forward: BF16 input, FP32 normalisation; retained: NVFP4 output
//                  and the FP32 per-token statistic; backward: FP32 reconstruction
//                  and reduction, BF16 gradient.
//   SiLU-multiply  forward: BF16 gate/up inputs, FP32 arithmetic; retained:
//                  separate NVFP4 gate/up copies; backward: FP32 reconstruction and
//                  derivatives, BF16 gradients.
// The abstract adds that forward nonlinear ops read BF16 (never dequantised
// NVFP4) inputs, and that the RMSNorm output is quantised once and reused by the
// following projections.
//
// Quantising a tensor needs its global amax first, so each fused quantiser runs
// two passes: pass 1 computes the statistic/activation and its amax, pass 2
// recomputes the FP32 values (re-reading the input, mostly from L2) and encodes.
#include <algorithm>

#include "common.cuh"
#include "encode_tiles.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pact {

// ============================================================== RMSNorm forward
// Both passes stream whole rows through a per-warp ring of shared-memory slots,
// filled by bulk asynchronous copies (one per row, issued by lane 0 and completed
// on the slot's mbarrier), so every warp keeps several rows in flight while it
// works on one, with few registers.  gamma is staged once per CTA.  Lane l owns
// blocks l, l+32, ... (BPL of them) of a row.
constexpr uint64_t kRowWaitNs = 2000000000ull;  // 2 s per ring wait

struct RowRing {
  uint32_t data;   // shared address of this warp's slot 0
  uint32_t bars;   // shared address of this warp's barrier 0
  uint32_t bytes;  // bytes of one row (one slot)
  int ns;          // slots
};

// Lane 0 issues the copy of row `row` (bytes at src) into slot k.
__device__ __forceinline__ void ring_issue(const RowRing& rr, int k, const void* src) {
  mbar_expect_tx(rr.bars + 8u * k, rr.bytes);
  bulk_load(rr.data + (uint32_t)k * rr.bytes, src, rr.bytes, rr.bars + 8u * k);
}

// Dynamic shared memory of a row-ring kernel: [gamma (padded to 128)] [warps x ns
// slots] [warps x ns barriers].  Three CTAs share an SM when at least four warps
// with two slots each fit in 66 KB: the statistic's per-lane sums are serial
// chains, so more warps beat deeper rings (on GB300 at H = 3072, 3 CTAs of 4 warps
// with 2 slots ran 10-15 % faster than 1 CTA of 8 warps with 4 slots).  Wider rows
// take one CTA per SM within 200 KB.
struct RingShape {
  int warps, ns, ctas_per_sm;
  size_t smem;
};
static RingShape ring_shape(int64_t H, int copies_per_row, bool with_gamma) {
  const size_t row = (size_t)H * 2 * copies_per_row;
  const size_t fixed = with_gamma ? (size_t)((H * 2 + 127) / 128 * 128) : 0;
  RingShape r;
  r.ctas_per_sm = fixed + 8 * row <= 66 * 1024 ? 3 : 1;
  const size_t avail = (r.ctas_per_sm == 3 ? 66 : 200) * 1024 - fixed;
  r.warps = (int)std::min<size_t>(8, std::max<size_t>(1, avail / (2 * row)));
  r.ns = (int)std::min<size_t>(4, std::max<size_t>(2, avail / (r.warps * row)));
  r.smem = fixed + (size_t)r.warps * r.ns * row + (size_t)r.warps * r.ns * 8 + 128;
  return r;
}

__device__ __forceinline__ void stage_gamma(uint8_t* sm, const uint16_t* gamma, int64_t H) {
  for (int i = threadIdx.x; i < (int)(H >> 3); i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = reinterpret_cast<const uint4*>(gamma)[i];
}

// Set up this warp's ring (barriers by lane 0) and return it.  The caller syncs the
// CTA before the first copy.
__device__ __forceinline__ RowRing ring_setup(uint8_t* sm, uint32_t base_off, int64_t H,
                                              int copies, int ns) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  RowRing rr;
  rr.bytes = (uint32_t)(H * 2 * copies);
  rr.ns = ns;
  rr.data = smem_addr(sm) + base_off + (uint32_t)(warp * ns) * rr.bytes;
  rr.bars = smem_addr(sm) + base_off + (uint32_t)(nw * ns) * rr.bytes + 8u * (uint32_t)(warp * ns);
  if ((threadIdx.x & 31) == 0) {
    for (int k = 0; k < ns; ++k) mbar_init(rr.bars + 8u * k, 1);
    fence_mbar_init();
  }
  return rr;
}

// Before a CTA leaves after a timeout: let this warp's copies still in flight land
// (bounded), so no copy writes shared memory that another CTA may own next.
__device__ __forceinline__ void ring_drain(const RowRing& rr, uint32_t pending, uint32_t phases) {
  for (int k = 0; k < rr.ns; ++k)
    if (pending & (1u << k)) mbar_wait(rr.bars + 8u * k, (phases >> k) & 1u, 10000000ull, nullptr);
}

// Pass 1: per row, rstd in the fixed order (sum of squares block by block, element
// by element, per lane; then a butterfly over offsets 16, 8, 4, 2, 1; the oracle's
// order) and max |y| of y = RN(RN(x rstd) gamma), folded into *amax_bits.
template <int BPL>
__global__ void __launch_bounds__(256) k_rmsnorm_stat(const uint16_t* __restrict__ x,
                                                      const uint16_t* __restrict__ gamma,
                                                      int64_t M, int64_t H, float eps, int ns,
                                                      float* __restrict__ rstd,
                                                      unsigned* __restrict__ amax_bits,
                                                      unsigned* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t sm[];
  const int lane = threadIdx.x & 31;
  const int nb = (int)(H >> 4);
  const uint32_t goff = (uint32_t)((H * 2 + 127) / 128 * 128);
  stage_gamma(sm, gamma, H);
  const RowRing rr = ring_setup(sm, goff, H, 1, ns);
  __syncthreads();
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t step = (int64_t)gridDim.x * (blockDim.x >> 5);
  uint32_t pending = 0, phases = 0;
  if (lane == 0)
    for (int k = 0; k < ns; ++k) {
      const int64_t r = wid + k * step;
      if (r < M) {
        ring_issue(rr, k, x + r * H);
        pending |= 1u << k;
      }
    }
  uint32_t amax = 0;
  int k = 0;
  uint32_t par = 0;
  for (int64_t row = wid; row < M; row += step) {
    // every lane observes the copy's completion; the decision to give up is the warp's
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(rr.bars + 8u * k, par, kRowWaitNs, nullptr))) {
      if (lane == 0) {
        atomicOr(status, PACT_DEV_TIMEOUT);
        ring_drain(rr, pending, phases);
      }
      break;
    }
    const uint8_t* slot = sm + (rr.data - smem_addr(sm)) + (uint32_t)k * rr.bytes;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      const int b = lane + 32 * j;
      if (b < nb) {
        float f[16];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(slot + 32 * b), f);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(slot + 32 * b + 16), f + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc = __fadd_rn(acc, __fmul_rn(f[i], f[i]));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
      acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
    const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, (float)H), eps)));
    if (lane == 0 && PACT_IN(row < M)) rstd[row] = rs;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      const int b = lane + 32 * j;
      if (b < nb) {
        float f[16], gm[16];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(slot + 32 * b), f);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(slot + 32 * b + 16), f + 8);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sm + 32 * b), gm);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sm + 32 * b + 16), gm + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float y = __fmul_rn(__fmul_rn(f[i], rs), gm[i]);
          PACT_NAN_F32(y);
          amax = max(amax, __float_as_uint(y) & 0x7FFFFFFFu);
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      pending &= ~(1u << k);
      const int64_t nr = row + (int64_t)ns * step;
      if (nr < M) {
        fence_proxy_async_smem();  // the slot's reads are done before the copy refills it
        ring_issue(rr, k, x + nr * H);
        pending |= 1u << k;
        phases ^= 1u << k;
      }
    }
    if (++k == ns) {
      k = 0;
      par ^= 1u;
    }
  }
  block_max_atomic(amax, amax_bits);
}

// Pass 2: y recomputed from x (read again, mostly from L2) and the stored rstd, then
// encoded, through the shared tile encoder (encode_tiles.cuh): x arrives in 32-row x
// 64-column TMA tiles, a lane takes four blocks of one row, gamma comes through L1
// (every lane of a warp reads the same 64 values of a tile) and rstd once per tile.
struct RmsNormValues {
  const uint16_t* gamma;
  const float* rstd;
  float rs;
  __device__ __forceinline__ void row(uint32_t r) { rs = __ldg(rstd + r); }
  __device__ __forceinline__ uint32_t block(const uint4& a, const uint4& b, uint32_t col,
                                            float* f) {
    const uint4* gp = reinterpret_cast<const uint4*>(gamma + col);
    float gm[16];
    bf16x8_to_f32(a, f);
    bf16x8_to_f32(b, f + 8);
    bf16x8_to_f32(__ldg(gp), gm);
    bf16x8_to_f32(__ldg(gp + 1), gm + 8);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      f[i] = __fmul_rn(__fmul_rn(f[i], rs), gm[i]);
      am = fmaxf(am, fabsf(f[i]));
    }
    return __float_as_uint(am);
  }
  __device__ __forceinline__ float elem(const uint4& a, uint32_t i, uint32_t col) {
    const float gi = __uint_as_float((uint32_t)__ldg(gamma + col + i) << 16);
    return __fmul_rn(__fmul_rn(bf16x8_at(a, i), rs), gi);
  }
};

__global__ void __launch_bounds__(kTileThreads, 2) k_rmsnorm_encode(
    const __grid_constant__ CUtensorMap tmx, const uint16_t* __restrict__ gamma,
    const float* __restrict__ rstd, int64_t M, int64_t H, int64_t Mpad, FastDiv upr_div,
    const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    float* __restrict__ g_out, unsigned* __restrict__ status) {
  extern __shared__ uint8_t esm[];
  const TensorScale ts = tensor_scale(__uint_as_float(*amax_bits));
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = ts.g;
  RmsNormValues op{gamma, rstd, 0.0f};
  encode_tiles(&tmx, M, H, Mpad, upr_div, ts, codes, sf, status, esm, op);
}

// ============================================================== SiLU-multiply
// The exact h of element i (0..15) of a block held as two uint4 of BF16 gate and
// up values, for a runtime i, without indexing a register array.  Called from
// loops that are not unrolled: the exact recipe is long, and copies of it for
// every element would not fit the instruction cache.
__device__ __forceinline__ float silu_exact_at(const uint4& g0, const uint4& g1, const uint4& u0,
                                               const uint4& u1, int i) {
  auto word = [](const uint4& a, const uint4& b, int i) {
    const uint4& v = i < 8 ? a : b;
    const int k = (i & 7) >> 1;
    const uint32_t w = k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
    return (i & 1) ? (w & 0xFFFF0000u) : (w << 16);
  };
  return silu_mul(__uint_as_float(word(g0, g1, i)), __uint_as_float(word(u0, u1, i)));
}

// Fast h for a block of 16 (gate values gf, up values uf) and its largest
// magnitude.  The fast values are used only where silu_mul_fast's bound is
// guaranteed for the whole block: every |gate| zero or in [2^-60, 80], every
// input finite, and the block maximum between 2^-100 and 2^100;
// silu_block_fast_ok says whether it is.
__device__ __forceinline__ float silu_block_fast(const float* gf, const float* uf, float* hf) {
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float2 h = silu_mul_fast2(make_float2(gf[i], gf[i + 1]), make_float2(uf[i], uf[i + 1]));
    hf[i] = h.x;
    hf[i + 1] = h.y;
    am = fmaxf(am, fmaxf(fabsf(h.x), fabsf(h.y)));
  }
  return am;
}
__device__ __forceinline__ bool silu_block_fast_ok(uint32_t gmax_bits, uint32_t umax_bits,
                                                   bool tiny_gate, float am) {
  return gmax_bits <= 0x42A00000u /* 80.0f */ && umax_bits < 0x7F800000u && !tiny_gate &&
         am >= 0x1p-100f && am <= 0x1p+100f;
}
// Whether some gate value of the 8 BF16 values is nonzero but below 2^-60: there
// g / (1 + exp(-g)) may leave the normal range and the fast quotient its bound,
// while a large up value can still lift h far above the block's rounding
// thresholds.  With every |g| zero or in [2^-60, 80] that quotient is zero or
// normal.
__device__ __forceinline__ bool bf16x8_has_tiny(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool t = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
    t |= (lo - 1u) < (0x2180u - 1u);  // 0 < |x| < 2^-60 (bf16 bits of 2^-60: 0x2180)
    t |= (hi - 1u) < (0x2180u - 1u);
  }
  return t;
}

// Pass 1: amax of h = silu(gate) * up, of gate and of up.  The exact recipe runs
// only for blocks that may hold the maximum.  Each round the warp takes A, the
// largest of its running value am and every lane's block maximum of fast values
// (am_blk), and a lane evaluates its block exactly only if am_blk >= A (1 - 3r)
// (r = kSiluRel); the block behind A always is, so A stays the fast value of an
// exactly evaluated element y.  A block skipped this way holds nothing above
// exact(y): exact <= fast (1 + r) < A (1 - 3r)(1 + r) < A (1 - 2r) <= exact(y), and
// y's lane keeps exact(y) in its maximum.  So the largest exact value over the
// evaluated blocks is the exact maximum, and only a few blocks per warp take the
// exact path.  A block outside the fast bound is always evaluated exactly (its
// exact maximum then enters A).  The loop advances by warps so that every lane
// takes part in each round.
__global__ void __launch_bounds__(256, 3) k_silu_amax(const uint16_t* __restrict__ gu, int64_t M,
                                                      int64_t I, FastDiv bpr_div,
                                                      unsigned* __restrict__ amax3) {
  const uint32_t bpr = (uint32_t)(I >> 4);
  const uint32_t total = (uint32_t)M * bpr;
  const uint32_t lane = threadIdx.x & 31u;
  const float keep = 1.0f - 3.0f * kSiluRel;
  uint32_t ah = 0, ag = 0, au = 0;
  float am = 0.0f;
  const uint32_t stride = gridDim.x * blockDim.x;
  // the next round's 64 bytes are loaded before this one is processed
  uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0, n2 = n0, n3 = n0;
  auto fetch = [&](uint32_t it) {
    if (it < total) {
      const int64_t row = bpr_div.div(it), b = it - (uint32_t)row * bpr;
      const uint4* gp = reinterpret_cast<const uint4*>(gu + row * 2 * I + b * 16);
      const uint4* up = reinterpret_cast<const uint4*>(gu + row * 2 * I + I + b * 16);
      n0 = ldg_stream(gp);
      n1 = ldg_stream(gp + 1);
      n2 = ldg_stream(up);
      n3 = ldg_stream(up + 1);
    }
  };
  const uint32_t first = blockIdx.x * blockDim.x + (threadIdx.x & ~31u);
  fetch(first + lane);
  for (uint32_t w0 = first; w0 < total; w0 += stride) {
    const uint32_t it = w0 + lane;
    const bool act = it < total;
    const uint4 g0 = n0, g1 = n1, u0 = n2, u1 = n3;
    fetch(it + stride);
    const uint32_t gb = max(absmax_bf16x8_bits(g0), absmax_bf16x8_bits(g1));
    const uint32_t ub = max(absmax_bf16x8_bits(u0), absmax_bf16x8_bits(u1));
    float am_blk = 0.0f;
    bool ok = true;
    float hf[16];
    if (act) {
      ag = max(ag, gb);
      au = max(au, ub);
      float gf[16], uf[16];
      bf16x8_to_f32(g0, gf);
      bf16x8_to_f32(g1, gf + 8);
      bf16x8_to_f32(u0, uf);
      bf16x8_to_f32(u1, uf + 8);
      am_blk = silu_block_fast(gf, uf, hf);
      ok = silu_block_fast_ok(gb, ub, bf16x8_has_tiny(g0) || bf16x8_has_tiny(g1), am_blk);
    }
    float A = fmaxf(am, ok ? am_blk : 0.0f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) A = fmaxf(A, __shfl_xor_sync(0xFFFFFFFFu, A, off));
    float em = 0.0f;
    if (act && (!ok || !(am_blk < A * keep))) {
      // the elements that may reach A (every element of a block outside the bound)
      uint32_t cand = 0xFFFFu;
      if (ok) {
        cand = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) cand |= (fabsf(hf[i]) < A * keep ? 0u : 1u) << i;
      }
      while (cand) {
        const int i = __ffs(cand) - 1;
        cand &= cand - 1;
        const uint32_t xb = __float_as_uint(silu_exact_at(g0, g1, u0, u1, i)) & 0x7FFFFFFFu;
        ah = max(ah, xb);
        if (xb < 0x7F800000u) em = fmaxf(em, __uint_as_float(xb));
      }
    }
    // a block outside the fast bound enters the running value with its exact maximum
    float B = ok ? 0.0f : em;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) B = fmaxf(B, __shfl_xor_sync(0xFFFFFFFFu, B, off));
    am = fmaxf(A, B);
  }
  block_max_atomic(ah, amax3 + 0);
  block_max_atomic(ag, amax3 + 1);
  block_max_atomic(au, amax3 + 2);
}

// Pass 2: one thread per block of 16 columns of one row; encodes h, gate and up.
// Fast values give the exact encoding of h wherever both roundings are certain:
// the block scale when e4m3 of the fast block maximum over d, widened by
// (1 -/+ 2r), rounds to one code; an element's code e2m1(RN(h / t)) when the fast
// value times fl = RN(rlo (1 - 2r)) and times fh = RN(rhi (1 + 2r)) round to one
// E2M1 code.  With |h - fast| <= 2^-20.5 |h| and rlo < 1/t < rhi, the rounded
// products bound |h| / t from both sides (each adds at most two roundings of
// 2^-24 to a widening of 2r = 2^-17), and both roundings to FP32 and to E2M1 are
// monotonic.  Elements that fail the second test are encoded from their exact
// values; a block that fails the first, or lies outside the fast bound, is encoded
// from exact values throughout.
struct SiluOut {
  uint8_t* codes[3];
  uint8_t* sf[3];
  float* g[3];
};

__global__ void __launch_bounds__(256, 3) k_silu_encode(const uint16_t* __restrict__ gu,
                                                        int64_t M, int64_t Mpad, int64_t I,
                                                        FastDiv bpr_div,
                                                        const float* __restrict__ amax3_opt,
                                                        const unsigned* __restrict__ amax3,
                                                        SiluOut out) {
  TensorScale ts[3];
  __shared__ float2 brk[3][256];  // bracket tables of the h, gate and up scales
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    ts[k] = tensor_scale(amax3_opt ? amax3_opt[k] : __uint_as_float(amax3[k]));
    if (blockIdx.x == 0 && threadIdx.x == 0) *out.g[k] = ts[k].g;
    brk[k][threadIdx.x] = bracket_entry(threadIdx.x, ts[k].g);  // blockDim.x == 256
  }
  __syncthreads();
  const float lo_f = 1.0f - 2.0f * kSiluRel, hi_f = 1.0f + 2.0f * kSiluRel;
  const float rcp_d = ts[0].rcp_d;
  const uint32_t bpr = (uint32_t)(I >> 4);
  const uint32_t total = (uint32_t)Mpad * bpr;
  const uint32_t stride = gridDim.x * blockDim.x;
  // the next iteration's 64 bytes are loaded before this one is processed
  uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0, n2 = n0, n3 = n0;
  auto fetch = [&](uint32_t it) {
    if (it < total) {
      const int64_t row = bpr_div.div(it), b = it - (uint32_t)row * bpr;
      if (row < M) {
        const uint4* gp = reinterpret_cast<const uint4*>(gu + row * 2 * I + b * 16);
        const uint4* up = reinterpret_cast<const uint4*>(gu + row * 2 * I + I + b * 16);
        n0 = ldg_stream(gp);
        n1 = ldg_stream(gp + 1);
        n2 = ldg_stream(up);
        n3 = ldg_stream(up + 1);
      }
    }
  };
  fetch(blockIdx.x * blockDim.x + threadIdx.x);
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += stride) {
    const uint4 g0 = n0, g1 = n1, u0 = n2, u1 = n3;
    fetch(it + stride);
    const int64_t row = bpr_div.div(it), b = it - (uint32_t)row * bpr;
    const int64_t so = sf_offset(row, b, bpr);
    if (!PACT_IN(so < Mpad * (int64_t)bpr)) continue;
    if (row >= M) {
#pragma unroll
      for (int k = 0; k < 3; ++k) out.sf[k][so] = 0;
      continue;
    }
    const uint32_t gb = absmax_bf16x16_bits(g0, g1), ub = absmax_bf16x16_bits(u0, u1);
    // gate and up (their BF16 values are exact) and the fast h, from one unpack
    uint32_t wg[2], wu[2], dg[2], du[2], wh[2], dh[2];
    const uint32_t sg = scale_byte(__uint_as_float(gb), ts[1]);
    const uint32_t su = scale_byte(__uint_as_float(ub), ts[2]);
    float hf[16], am_blk;
    {
      float gf[16], uf[16];
      bf16x8_to_f32(g0, gf);
      bf16x8_to_f32(g1, gf + 8);
      bf16x8_to_f32(u0, uf);
      bf16x8_to_f32(u1, uf + 8);
      am_blk = silu_block_fast(gf, uf, hf);
      codes16(gf, brk[1][sg], wg[0], wg[1], dg[0], dg[1]);
      codes16(uf, brk[2][su], wu[0], wu[1], du[0], du[1]);
    }
    // ---- h: scale and codes from the fast values where both roundings are certain
    bool fast = silu_block_fast_ok(gb, ub, bf16x8_has_tiny(g0) || bf16x8_has_tiny(g1), am_blk) &&
                ts[0].g > 0.0f && rcp_d > 0.0f;
    uint32_t sh = 0;
    if (fast) {
      const float q = __fmul_rn(am_blk, rcp_d);
      uint16_t pr;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
          : "=h"(pr)
          : "f"(__fmul_rn(q, hi_f)), "f"(__fmul_rn(q, lo_f)));
      sh = pr & 0xFFu;
      fast = sh == (uint32_t)(pr >> 8);
    }
    float2 br = brk[0][sh];
    const float fl = __fmul_rn(br.x, lo_f), fh = __fmul_rn(br.y, hi_f);
    fast = fast && br.x > 0.0f && fh <= 3.4028234663852886e38f;
    float th;  // the decode step of h's block
    if (fast) {
      wh[0] = e2m1x8_of_products(hf, fl);
      wh[1] = e2m1x8_of_products(hf + 8, fl);
      dh[0] = wh[0] ^ e2m1x8_of_products(hf, fh);
      dh[1] = wh[1] ^ e2m1x8_of_products(hf + 8, fh);
      th = __fmul_rn(e4m3_to_f32(sh), ts[0].g);
    } else {
      // the exact block maximum and scale; every code from its exact value below
      uint32_t em = 0;
#pragma unroll 1
      for (int i = 0; i < 16; ++i)
        em = max(em, __float_as_uint(silu_exact_at(g0, g1, u0, u1, i)) & 0x7FFFFFFFu);
      BlockStep st;
      sh = block_scale_fast(__uint_as_float(em), ts[0], &st);
      th = st.t;
      wh[0] = wh[1] = 0u;
      dh[0] = dh[1] = 0xFFFFFFFFu;  // every element
    }
    // the rare elements whose code the fast values leave open: exact h
    if (dh[0] | dh[1]) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll 1
        while (dh[q]) {
          const uint32_t sh4 = ((uint32_t)__ffs(dh[q]) - 1u) & ~3u;
          dh[q] &= ~(0xFu << sh4);
          const uint32_t c =
              e2m1_code_exact(silu_exact_at(g0, g1, u0, u1, 8 * q + (int)(sh4 >> 2)), th);
          wh[q] = (wh[q] & ~(0xFu << sh4)) | (c << sh4);
        }
      }
    }
    if (dg[0] | dg[1] | du[0] | du[1]) {
      const float tg = __fmul_rn(e4m3_to_f32(sg), ts[1].g);
      const float tu = __fmul_rn(e4m3_to_f32(su), ts[2].g);
      wg[0] = fix_word(wg[0], dg[0], tg, [&](uint32_t i) { return bf16x8_at(g0, i); });
      wg[1] = fix_word(wg[1], dg[1], tg, [&](uint32_t i) { return bf16x8_at(g1, i); });
      wu[0] = fix_word(wu[0], du[0], tu, [&](uint32_t i) { return bf16x8_at(u0, i); });
      wu[1] = fix_word(wu[1], du[1], tu, [&](uint32_t i) { return bf16x8_at(u1, i); });
    }
    const int64_t co = row * (I >> 1) + b * 8;
    *reinterpret_cast<uint2*>(out.codes[0] + co) = make_uint2(wh[0], wh[1]);
    *reinterpret_cast<uint2*>(out.codes[1] + co) = make_uint2(wg[0], wg[1]);
    *reinterpret_cast<uint2*>(out.codes[2] + co) = make_uint2(wu[0], wu[1]);
    out.sf[0][so] = (uint8_t)sh;
    out.sf[1][so] = (uint8_t)sg;
    out.sf[2][so] = (uint8_t)su;
  }
}

// ============================================================== backward kernels
// SiLU-multiply backward; one thread per block of 16 columns, the next block's
// codes, scales and dh in flight while the current one is processed; the amax of the
// BF16 outputs folds in packed (max.xorsign.abs on BF16 pairs, signs masked at the
// end).  On GB300 the prefetch and the packed amax took it from 96 to 87 us at
// 8192 x 8192 (0.80 of the measured HBM copy bandwidth).
__global__ void __launch_bounds__(256) k_silu_bwd(
    const uint8_t* __restrict__ gc, const uint8_t* __restrict__ gsf, const float* __restrict__ gg,
    const uint8_t* __restrict__ uc, const uint8_t* __restrict__ usf, const float* __restrict__ ug,
    const uint16_t* __restrict__ dh, int64_t M, int64_t I, FastDiv bpr_div,
    uint16_t* __restrict__ dgu, unsigned* __restrict__ out_amax) {
  const uint32_t bpr = (uint32_t)(I >> 4);
  const uint32_t total = (uint32_t)M * bpr;
  const float g_gate = *gg, g_up = *ug;
  uint32_t amax = 0;
  // the next block's inputs are loaded before this one is processed
  uint2 ncg = make_uint2(0u, 0u), ncu = ncg;
  uint32_t nsg = 0, nsu = 0;
  uint4 nd0 = make_uint4(0u, 0u, 0u, 0u), nd1 = nd0;
  auto fetch = [&](uint32_t it) {
    if (it < total) {
      const int64_t row = bpr_div.div(it), b = it - (uint32_t)row * bpr;
      const int64_t so = sf_offset(row, b, bpr);
      ncg = *reinterpret_cast<const uint2*>(gc + row * (I >> 1) + b * 8);
      ncu = *reinterpret_cast<const uint2*>(uc + row * (I >> 1) + b * 8);
      nsg = gsf[so];
      nsu = usf[so];
      const uint4* dp = reinterpret_cast<const uint4*>(dh + row * I + b * 16);
      nd0 = ldg_stream(dp);
      nd1 = ldg_stream(dp + 1);
    }
  };
  const uint32_t stride = gridDim.x * blockDim.x;
  fetch(blockIdx.x * blockDim.x + threadIdx.x);
  uint32_t am2 = 0;  // packed max |.| of the BF16 outputs (sign bits masked at the end)
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += stride) {
    const uint2 cg = ncg, cu = ncu;
    const uint32_t sg0 = nsg, su0 = nsu;
    const uint4 d0 = nd0, d1 = nd1;
    fetch(it + stride);
    const int64_t row = bpr_div.div(it), b = it - (uint32_t)row * bpr;
    float gv[16], uv[16], d[16];
    dequant16_f32(cg, e4m3_to_f32(sg0) * g_gate, gv);
    dequant16_f32(cu, e4m3_to_f32(su0) * g_up, uv);
    bf16x8_to_f32(d0, d);
    bf16x8_to_f32(d1, d + 8);
    uint32_t og[8], ou[8];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float rg[2], ru[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        // tolerance-checked BF16 gradient: fast exp and division are enough here
        const float gk = gv[i + k], uk = uv[i + k], dk = d[i + k];
        const float sg = __fdividef(1.0f, 1.0f + __expf(-gk));
        const float dsilu = sg * fmaf(gk, 1.0f - sg, 1.0f);
        rg[k] = (dk * uk) * dsilu;
        ru[k] = dk * (gk * sg);
      }
      og[i / 2] = pack_bf16x2(rg[0], rg[1]);
      ou[i / 2] = pack_bf16x2(ru[0], ru[1]);
      uint32_t t;
      asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(og[i / 2]), "r"(ou[i / 2]));
      asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(am2) : "r"(am2), "r"(t));
    }
    if (!PACT_IN(row < M && b < bpr)) continue;
#pragma unroll
    for (int i = 0; i < 8; ++i) PACT_NAN_BF16X2(og[i]), PACT_NAN_BF16X2(ou[i]);
    uint4* pg = reinterpret_cast<uint4*>(dgu + row * 2 * I + b * 16);
    uint4* pu = reinterpret_cast<uint4*>(dgu + row * 2 * I + I + b * 16);
    pg[0] = make_uint4(og[0], og[1], og[2], og[3]);
    pg[1] = make_uint4(og[4], og[5], og[6], og[7]);
    pu[0] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    pu[1] = make_uint4(ou[4], ou[5], ou[6], ou[7]);
  }
  am2 &= 0x7FFF7FFFu;
  amax = max(amax, max(am2 << 16, am2 & 0xFFFF0000u));
  if (out_amax) block_max_atomic(amax, out_amax);
}

// RMSNorm backward; one warp per row, lane l owns blocks l, l+32, ...
// n = yhat / gamma, dn = dy * gamma, c = sum(dn * n) / H, dx = rstd (dn - n c) [+ dres].
template <int BPL>
__global__ void __launch_bounds__(256) k_rmsnorm_bwd(
    const uint8_t* __restrict__ yc, const uint8_t* __restrict__ ysf, const float* __restrict__ yg,
    const uint16_t* __restrict__ gamma, const float* __restrict__ rstd,
    const uint16_t* __restrict__ dy, const uint16_t* dres, int64_t M, int64_t H,
    uint16_t* dx, unsigned* __restrict__ out_amax) {
  // The row's codes, scales and dy stay in registers between the reduction and the
  // output pass.  sum(dn * n) = sum(dy * gamma * yhat / gamma) = sum(dy * yhat), so
  // the reduction needs no division; the output pass divides by gamma with the
  // fast approximate division (the result is a tolerance-checked BF16 gradient).
  const int lane = threadIdx.x & 31;
  const int nb = (int)(H >> 4);
  const float g = *yg;
  uint32_t amax = 0;  // max |dx| over this thread's outputs, as FP32 bits of the BF16 values
  uint32_t am2 = 0;   // the same, packed (max.xorsign.abs on BF16 pairs, signs masked at the end)
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < M;
       row += (int64_t)gridDim.x * 8) {
    uint2 cw[BPL];
    uint32_t sb[BPL];
    uint4 dv[BPL][2];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      const int b = lane + 32 * j;
      if (b < nb) {
        cw[j] = *reinterpret_cast<const uint2*>(yc + row * (H >> 1) + b * 8);
        sb[j] = ysf[sf_offset(row, b, nb)];
        const uint4* dp = reinterpret_cast<const uint4*>(dy + row * H + b * 16);
        dv[j][0] = ldg_stream(dp);
        dv[j][1] = ldg_stream(dp + 1);
      }
    }
    float dot = 0.0f;
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      if (lane + 32 * j < nb) {
        float yv[16], d[16];
        dequant16_f32(cw[j], e4m3_to_f32(sb[j]) * g, yv);
        bf16x8_to_f32(dv[j][0], d);
        bf16x8_to_f32(dv[j][1], d + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) dot = fmaf(d[i], yv[i], dot);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    const float c = dot / (float)H;
    const float rs = rstd[row];
#pragma unroll
    for (int j = 0; j < BPL; ++j) {
      const int b = lane + 32 * j;
      if (b < nb) {
        float yv[16], gm[16], d[16], r[16];
        dequant16_f32(cw[j], e4m3_to_f32(sb[j]) * g, yv);
        const uint4* gp = reinterpret_cast<const uint4*>(gamma + b * 16);
        bf16x8_to_f32(__ldg(gp), gm);
        bf16x8_to_f32(__ldg(gp + 1), gm + 8);
        bf16x8_to_f32(dv[j][0], d);
        bf16x8_to_f32(dv[j][1], d + 8);
        if (dres) {
          const uint4* rp = reinterpret_cast<const uint4*>(dres + row * H + b * 16);
          bf16x8_to_f32(rp[0], r);
          bf16x8_to_f32(rp[1], r + 8);
        }
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float v[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float n = __fdividef(yv[i + k], gm[i + k]);
            v[k] = rs * fmaf(d[i + k], gm[i + k], -n * c);
            if (dres) v[k] += r[i + k];
          }
          o[i / 2] = pack_bf16x2(v[0], v[1]);
          asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(am2) : "r"(am2), "r"(o[i / 2]));
        }
        uint4* op = reinterpret_cast<uint4*>(dx + row * H + b * 16);
        if (!PACT_IN(row < M && b < nb)) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) PACT_NAN_BF16X2(o[i]);
        op[0] = make_uint4(o[0], o[1], o[2], o[3]);
        op[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
  am2 &= 0x7FFF7FFFu;
  amax = max(amax, max(am2 << 16, am2 & 0xFFFF0000u));
  if (out_amax) block_max_atomic(amax, out_amax);
}

__global__ void k_pexp(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = pexp(x[i]);
}

// ============================================================== launchers
static int blocks_for(int64_t work, int threads, int cap) {
  int64_t b = (work + threads - 1) / threads;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

template <typename F>
static cudaError_t dispatch_bpl(int64_t H, F&& f) {
  const int bpl = (int)(((H >> 4) + 31) / 32);
  switch (bpl) {
    case 1: return f(std::integral_constant<int, 1>());
    case 2: return f(std::integral_constant<int, 2>());
    case 3: return f(std::integral_constant<int, 3>());
    case 4: return f(std::integral_constant<int, 4>());
    case 5: case 6: return f(std::integral_constant<int, 6>());
    case 7: case 8: return f(std::integral_constant<int, 8>());
    case 9: case 10: case 11: case 12: return f(std::integral_constant<int, 12>());
    case 13: case 14: case 15: case 16: return f(std::integral_constant<int, 16>());
    case 17: case 18: case 19: case 20: case 21: case 22: case 23: case 24:
      return f(std::integral_constant<int, 24>());
    default: return f(std::integral_constant<int, 32>());
  }
}

cudaError_t launch_rmsnorm_quant(const CUtensorMap& tmx, const uint16_t* x, const uint16_t* gamma, int64_t M,
                                 int64_t H, float eps, uint8_t* codes, uint8_t* sf, float* g,
                                 float* rstd, unsigned* ws_amax, unsigned* status, int num_sms,
                                 cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws_amax, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const int64_t Mpad = pad_to(M, 128);
  const RingShape rs = ring_shape(H, 1, true);
  e = dispatch_bpl(H, [&](auto bpl) {
    constexpr int BPL = decltype(bpl)::value;
    auto ks = k_rmsnorm_stat<BPL>;
    cudaError_t err = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)rs.smem);
    if (err != cudaSuccess) return err;
    note_launch();
    ks<<<blocks_for(M, rs.warps, num_sms * rs.ctas_per_sm), 32 * rs.warps, rs.smem, stream>>>(
        x, gamma, M, H, eps, rs.ns, rstd, ws_amax, status);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_rmsnorm_encode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tile_encode_smem_bytes());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t ntiles = (Mpad / 32) * (H / 64);
  note_launch();
  k_rmsnorm_encode<<<blocks_for(ntiles, kTileWarps, num_sms * 2), kTileThreads,
                     tile_encode_smem_bytes(), stream>>>(
      tmx, gamma, rstd, M, H, Mpad, FastDiv::make((uint32_t)(H / 64)), ws_amax, codes, sf, g,
      status);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_quant(const uint16_t* gateup, int64_t M, int64_t I,
                                  const float* amax3_opt, uint8_t* const codes[3],
                                  uint8_t* const sf[3], float* const g[3], unsigned* ws_amax3,
                                  int num_sms, cudaStream_t stream) {
  if (!amax3_opt) {
    cudaError_t e = cudaMemsetAsync(ws_amax3, 0, 3 * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    note_launch();
    k_silu_amax<<<blocks_for(M * (I / 16), 256, num_sms * 8), 256, 0, stream>>>(
        gateup, M, I, FastDiv::make((uint32_t)(I / 16)), ws_amax3);
  }
  SiluOut o;
  for (int k = 0; k < 3; ++k) {
    o.codes[k] = codes[k];
    o.sf[k] = sf[k];
    o.g[k] = g[k];
  }
  const int64_t Mpad = pad_to(M, 128);
  note_launch();
  k_silu_encode<<<blocks_for(Mpad * (I / 16), 256, num_sms * 16), 256, 0, stream>>>(
      gateup, M, Mpad, I, FastDiv::make((uint32_t)(I / 16)), amax3_opt, ws_amax3, o);
  return cudaGetLastError();
}

cudaError_t launch_silu_mul_bwd(const uint8_t* gc, const uint8_t* gsf, const float* gg,
                                const uint8_t* uc, const uint8_t* usf, const float* ug,
                                const uint16_t* dh, int64_t M, int64_t I, uint16_t* dgu,
                                unsigned* out_amax, int num_sms, cudaStream_t stream) {
  if (out_amax) {
    cudaError_t e = cudaMemsetAsync(out_amax, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
  }
  note_launch();
  k_silu_bwd<<<blocks_for(M * (I / 16), 256, num_sms * 16), 256, 0, stream>>>(
      gc, gsf, gg, uc, usf, ug, dh, M, I, FastDiv::make((uint32_t)(I / 16)), dgu, out_amax);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const uint8_t* yc, const uint8_t* ysf, const float* yg,
                               const uint16_t* gamma, const float* rstd, const uint16_t* dy,
                               const uint16_t* dres, int64_t M, int64_t H, uint16_t* dx,
                               unsigned* out_amax, int num_sms, cudaStream_t stream) {
  if (out_amax) {
    cudaError_t e = cudaMemsetAsync(out_amax, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
  }
  return dispatch_bpl(H, [&](auto bpl) {
    constexpr int BPL = decltype(bpl)::value;
    note_launch();
    k_rmsnorm_bwd<BPL><<<blocks_for(M, 8, num_sms * 8), 256, 0, stream>>>(
        yc, ysf, yg, gamma, rstd, dy, dres, M, H, dx, out_amax);
    return cudaGetLastError();
  });
}

cudaError_t launch_pexp(const float* x, float* y, int64_t n, cudaStream_t stream) {
  note_launch();
  k_pexp<<<blocks_for(n, 256, 4096), 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

}  // namespace pact
