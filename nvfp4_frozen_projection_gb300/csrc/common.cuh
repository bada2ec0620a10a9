// Device helpers shared by the libpact kernels (sm_103a only).
//
// NVFP4 (Table 6 of "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs"):
// E2M1 elements, one E4M3 scale per block of 16, plus an FP32 per-tensor scale.
// Conversions use the hardware cvt instructions (RN, satfinite); every FP32 step
// of the encode is an explicit __f*_rn intrinsic so the compiler cannot contract
// or reorder it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "status.h"

#if defined(__CUDA_ARCH__) && !defined(__CUDA_ARCH_FEAT_SM103_ALL)
#error "libpact kernels are written for sm_103a only"
#endif

namespace pact {

// ------------------------------------------------------------------ layout
__host__ __device__ __forceinline__ int64_t pad_to(int64_t x, int64_t m) {
  return (x + m - 1) / m * m;
}

// n / d for n < 2^31 by a multiply-high and a shift (Granlund and Montgomery's
// division by invariant integers): p = 31 + ceil(log2 d), m = ceil(2^p / d).
struct FastDiv {
  uint32_t d, m, s;
  __host__ static FastDiv make(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t p2 = 1ull << (31 + l);
    FastDiv f;
    f.d = d;
    f.m = (uint32_t)((p2 + d - 1) / d);
    f.s = l - 1;  // (n * m) >> (31 + l) == umulhi(n, m) >> (l - 1) for l >= 1
    return f;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return d == 1 ? n : (__umulhi(n, m) >> s);
  }
};

// Byte offset of the E4M3 scale of (row r, block c) in the 128x4-atom layout read
// by the block-scaled tensor-core MMA (c16p = pad4(cols/16)).
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t c16p) {
  return ((r >> 7) * (c16p >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 +
         (c & 3);
}

// Fused gate|up projection, interleaved forward layout: the output columns (the
// rows of the forward weight) are reordered in groups of 32, a group of gate
// columns then the matching group of up columns, so that one 32-column slice of an
// accumulator tile holds gate values and the next slice the up values of the same
// columns.  half = I, the width of each of gate and up.
__host__ __device__ __forceinline__ int64_t gu_logical(int64_t n, int64_t half) {
  const int64_t grp = n >> 6, j = n & 63;
  return j < 32 ? 32 * grp + j : half + 32 * grp + (j - 32);
}
__host__ __device__ __forceinline__ int64_t gu_interleaved(int64_t l, int64_t half) {
  return l < half ? 64 * (l >> 5) + (l & 31) : 64 * ((l - half) >> 5) + 32 + ((l - half) & 31);
}

// ------------------------------------------------------------------ codecs
// E4M3 (satfinite, RN) of a non-negative FP32 value -> byte.
__device__ __forceinline__ uint32_t e4m3_from_f32(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return (uint32_t)(r & 0xFFu);
}

// E4M3 byte -> FP32 (exact, through FP16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  uint16_t in = (uint16_t)(b & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// Two values -> E2M1 codes (RN, satfinite at 6): lo in bits 0..3, hi in bits 4..7.
// The sign bit follows the input, also when it rounds to zero (-0.1 -> 0x8,
// -0.0 -> 0x8; checked on GB300), matching the oracle's sign rule.
__device__ __forceinline__ uint32_t e2m1x2_mag(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t sign_bit(float x) { return __float_as_uint(x) >> 31; }

// Two E2M1 codes (one byte, first element in the low nibble) -> two floats, exact.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// Element encode of a block with decode step t = RN(e4m3(s) g):
//   q = e2m1_rne_satfinite(RN(x / t)),
// the quotient being one IEEE division.  A division per element is slow on the
// GPU, so the code is certified from two products instead.  Per block, rlo and rhi
// bracket 1/t: both are a hardware reciprocal estimate of t widened by 2^-19, and
// rlo t < 1 < rhi t is then verified exactly (the sign of a fused multiply-add),
// so the bracket holds whatever the estimate's error.  Then |x| rlo <= |x / t| <=
// |x| rhi, and rounding to FP32 and then to E2M1 are both monotonic, so when
// RN(x rlo) and RN(x rhi) give the same E2M1 code, RN(x / t) gives it too (a zero x
// gives the signed zero either way).  Only where the bracket straddles an E2M1
// rounding threshold is the code decided exactly without the products.  With BF16
// inputs that is about one element in 10^3: a BF16 value, an E4M3 scale and
// g = RN(amax / 2688) from a BF16 amax often put a quotient on a threshold up to
// the roundings of g and t, which is exactly where the division matters.  Blocks
// with t below 2^-96 (only in tensors whose amax is below about 2^-76) take the
// exact path throughout.
struct BlockStep {
  float t;    // decode step e4m3(s) * g
  float rlo;  // < 1/t, or 0 when the products may not be used
  float rhi;  // > 1/t, or 0 likewise
};

__device__ __forceinline__ float rcp_estimate(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ BlockStep block_step(float t) {
  BlockStep b;
  b.t = t;
  b.rlo = b.rhi = 0.0f;
  if (t >= 0x1p-96f && t <= 0x1p+125f) {
    const float r = rcp_estimate(t);
    const float lo = __fmul_rn(r, 1.0f - 0x1p-19f), hi = __fmul_rn(r, 1.0f + 0x1p-19f);
    if (__fmaf_rn(lo, t, -1.0f) < 0.0f && __fmaf_rn(hi, t, -1.0f) > 0.0f) {
      b.rlo = lo;
      b.rhi = hi;
    }
  }
  return b;
}

// Whether the products may certify codes for this block.
__device__ __forceinline__ bool step_certifiable(const BlockStep& b) { return b.rlo > 0.0f; }

// Magnitude code (0..7) of e2m1_rne_satfinite(RN(a / t)) for a >= 0 and t > 0,
// decided without dividing.  The E2M1 thresholds m (0.25, 0.75, 1.25, 1.75, 2.5,
// 3.5, 5) are FP32 values with an even significand, so RN(q) == m exactly when q
// lies in [m - hl, m + hh], hl and hh being half the FP32 spacing below and above
// m (ties at both ends go to the even m).  So RN(q) > m is a - (m + hh) t > 0, and
// RN(q) == m is a - (m - hl) t >= 0 as well, where the E2M1 rounding ties to the
// even code.  With D = RN(a - m t) from one fused multiply-add these are D > hh t
// and D >= -hl t: near the threshold (|a - m t| <= 2^-17 m t) a - m t is a
// multiple of at least a 2^-27 of a with at most ten significant bits, so D is
// exact; far from it |D| exceeds both hh t and hl t (at most 2^-23 m t), whose
// products are exact for t >= 2^-96.  A smaller t (and a, whose quotient is what
// matters) is first scaled by 2^64, exactly: t < 2^-96 forces g < 2^-87 and so
// a < 2^-75, far from overflow.
__device__ __forceinline__ bool e2m1_above(float a, float t, float mid, float hh) {
  return __fmaf_rn(-mid, t, a) > __fmul_rn(hh, t);
}
__device__ __forceinline__ bool e2m1_at(float a, float t, float mid, float hl) {
  return __fmaf_rn(-mid, t, a) >= -__fmul_rn(hl, t);
}
__device__ __forceinline__ uint32_t e2m1_mag_exact(float a, float t) {
  if (t < 0x1p-96f) {
    a = __fmul_rn(a, 0x1p+64f);
    t = __fmul_rn(t, 0x1p+64f);
  }
  // thresholds in increasing order; the first one that RN(q) does not exceed decides
  if (!e2m1_above(a, t, 0.25f, 0x1p-26f)) return 0u;  // a tie at 0.25 goes to 0 too
  if (!e2m1_above(a, t, 0.75f, 0x1p-25f)) return e2m1_at(a, t, 0.75f, 0x1p-25f) ? 2u : 1u;
  if (!e2m1_above(a, t, 1.25f, 0x1p-24f)) return 2u;  // a tie at 1.25 goes to 2
  if (!e2m1_above(a, t, 1.75f, 0x1p-24f)) return e2m1_at(a, t, 1.75f, 0x1p-24f) ? 4u : 3u;
  if (!e2m1_above(a, t, 2.5f, 0x1p-23f)) return 4u;   // a tie at 2.5 goes to 4
  if (!e2m1_above(a, t, 3.5f, 0x1p-23f)) return e2m1_at(a, t, 3.5f, 0x1p-23f) ? 6u : 5u;
  if (!e2m1_above(a, t, 5.0f, 0x1p-22f)) return 6u;   // a tie at 5 goes to 6
  return 7u;
}

// The code of one element, e2m1(RN(x / t)), by the exact decision above: a signed
// zero when t == 0 (a zero block or a zero tensor); the sign bit of a code is the
// sign bit of x, also when the value rounds to zero.
__device__ __forceinline__ uint32_t e2m1_code_exact(float x, float t) {
  const uint32_t sg = sign_bit(x) << 3;
  if (!(t > 0.0f)) return sg;
  return sg | e2m1_mag_exact(fabsf(x), t);
}

// Element i (runtime, 0..7) of eight register values, by a chain of selects: an
// indexed register array would move to local memory.
__device__ __forceinline__ float pick8(const float* x, uint32_t i) {
  float v = x[7];
#pragma unroll
  for (int k = 6; k >= 0; --k) v = (i == (uint32_t)k) ? x[k] : v;
  return v;
}

// Every code of a block whose products may not be used (t below 2^-96, or a failed
// bracket check): each code decided by e2m1_code_exact, in a loop that is not
// unrolled (the path is for tensors of tiny magnitude only).
__device__ __forceinline__ uint32_t codes8_exact(const float* x, float t) {
  uint32_t w = 0;
#pragma unroll 1
  for (uint32_t i = 0; i < 8; ++i) w |= e2m1_code_exact(pick8(x, i), t) << (4 * i);
  return w;
}

// Codes of a block with t == 0 (a zero block or a zero tensor): signed zeros.
__device__ __forceinline__ uint32_t codes8_signed_zero(const float* x) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) w |= (sign_bit(x[i]) << 3) << (4 * i);
  return w;
}

// Fix the codes where the bracket straddles a threshold.  For such an element the
// lower product gave magnitude code c and the upper c + 1, so the only threshold in
// question is m = (e2m1(c) + e2m1(c + 1)) / 2 (exact; from the hardware decode),
// and |x / t| is within 2^-18 m of it: the exact test of e2m1_mag_exact for that one
// threshold decides (hh = half the FP32 spacing above m, hl the same below, which is
// half of hh for m = 0.25, the one power of two among the thresholds).  The loop
// visits only the straddling elements (usually one): in a warp its cost is the
// largest count over the lanes, not the sum.
__device__ __forceinline__ uint32_t fix_straddles(uint32_t wl, uint32_t redo, const float* x,
                                                  float t) {
  uint32_t w = wl;
  // one bit per straddling element: bit 4i of redo | its neighbours folded down
  uint32_t bits = (redo | (redo >> 1) | (redo >> 2) | (redo >> 3)) & 0x11111111u;
#pragma unroll 1
  while (bits) {
    const uint32_t sh = (uint32_t)__ffs(bits) - 1u;  // 4 i
    bits &= bits - 1u;
    const float xi = pick8(x, sh >> 2);
    const uint32_t c = (wl >> sh) & 7u;
    const float2 d = e2m1x2_to_f32x2(c | ((c + 1u) << 4));
    const float m = __fmul_rn(__fadd_rn(d.x, d.y), 0.5f);
    const float hh = __int_as_float((__float_as_int(m) & 0x7F800000) - (24 << 23));
    const float hl = c == 0u ? __fmul_rn(hh, 0.5f) : hh;
    const float D = __fmaf_rn(-m, t, fabsf(xi));
    const uint32_t mag = D > __fmul_rn(hh, t) ? c + 1u : (D >= -__fmul_rn(hl, t) ? c + (c & 1u) : c);
    w = (w & ~(0xFu << sh)) | (((sign_bit(xi) << 3) | mag) << sh);
  }
  return w;
}

// RN(x * f) for 8 values -> 8 E2M1 codes packed in a uint32 (element 0 in bits
// 0..3).  The products are formed two at a time (mul.rn.f32x2 rounds each lane as
// mul.rn.f32 does) and the four code bytes are packed by one vector move.
__device__ __forceinline__ uint32_t e2m1x8_of_products(const float* x, float f) {
  uint32_t w;
  asm("{\n\t"
      ".reg .b64 rr, p0, p1, p2, p3;\n\t"
      ".reg .f32 q0, q1, q2, q3, q4, q5, q6, q7;\n\t"
      ".reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b64 rr, {%9, %9};\n\t"
      "mov.b64 p0, {%1, %2};\n\t"
      "mov.b64 p1, {%3, %4};\n\t"
      "mov.b64 p2, {%5, %6};\n\t"
      "mov.b64 p3, {%7, %8};\n\t"
      "mul.rn.f32x2 p0, p0, rr;\n\t"
      "mul.rn.f32x2 p1, p1, rr;\n\t"
      "mul.rn.f32x2 p2, p2, rr;\n\t"
      "mul.rn.f32x2 p3, p3, rr;\n\t"
      "mov.b64 {q0, q1}, p0;\n\t"
      "mov.b64 {q2, q3}, p1;\n\t"
      "mov.b64 {q4, q5}, p2;\n\t"
      "mov.b64 {q6, q7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, q1, q0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, q3, q2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, q5, q4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, q7, q6;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t"
      "}"
      : "=r"(w)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
        "f"(x[7]), "f"(f));
  return w;
}

// Encode 8 FP32 values of one block (element 0 in bits 0..3 of the result).
__device__ __forceinline__ uint32_t encode8(const float* x, const BlockStep& b) {
  if (!step_certifiable(b)) return b.t == 0.0f ? codes8_signed_zero(x) : codes8_exact(x, b.t);
  const uint32_t wl = e2m1x8_of_products(x, b.rlo);
  const uint32_t redo = wl ^ e2m1x8_of_products(x, b.rhi);
  if (redo == 0u) return wl;
  return fix_straddles(wl, redo, x, b.t);
}

// Dequantise one block of 16 codes (8 bytes) with decode step s = e4m3(scale) * g.
__device__ __forceinline__ void dequant16_f32(uint2 cw, float s, float* out) {
  const uint32_t w[2] = {cw.x, cw.y};
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 f = e2m1x2_to_f32x2((w[h] >> (8 * b)) & 0xFFu);
      out[8 * h + 2 * b] = f.x * s;
      out[8 * h + 2 * b + 1] = f.y * s;
    }
}

// Per-tensor scale, its block-scale divisor and that divisor's reciprocal.
struct TensorScale {
  float g;      // amax / 2688
  float d;      // 6 * g
  float rcp_d;  // RN(1 / d), or 0 when the fast block-scale quotient may not be used
};
__device__ __forceinline__ TensorScale tensor_scale(float amax) {
  TensorScale s;
  s.g = __fdiv_rn(amax, 2688.0f);
  s.d = __fmul_rn(6.0f, s.g);
  const float r = s.d > 0.0f ? __fdiv_rn(1.0f, s.d) : 0.0f;
  s.rcp_d = (r > 0.0f && r <= 3.4028234663852886e38f) ? r : 0.0f;
  return s;
}

// The decode step of scale byte s under the per-tensor scale g.
__device__ __forceinline__ BlockStep scale_step(uint32_t s, const TensorScale& ts) {
  return block_step(__fmul_rn(e4m3_to_f32(s), ts.g));
}

// Block scale byte s = e4m3(RN(amax_blk / d)) and the block's decode step, with the
// division itself (the offline weight pack).
__device__ __forceinline__ uint32_t block_scale(float amax_blk, const TensorScale& ts,
                                                BlockStep* st) {
  const uint32_t s = (ts.g == 0.0f) ? 0u : e4m3_from_f32(__fdiv_rn(amax_blk, ts.d));
  *st = scale_step(s, ts);
  return s;
}

// The same byte without a division per block: q = amax_blk * RN(1/d) is within
// 2^-22.4 of RN(amax_blk / d) (relative), so when q (1 - 2^-21) and q (1 + 2^-21)
// round to the same E4M3 byte, so does RN(amax_blk / d) (the rounding is
// monotonic); otherwise the division decides.  E4M3 thresholds lie at 2^-10 and
// above, so subnormal quotients never reach the check's margin.
__device__ __forceinline__ uint32_t block_scale_fast(float amax_blk, const TensorScale& ts,
                                                     BlockStep* st) {
  uint32_t s = 0;
  if (ts.g != 0.0f) {
    const float q = __fmul_rn(amax_blk, ts.rcp_d);
    s = e4m3_from_f32(__fmul_rn(q, 1.0f - 0x1p-21f));
    if (ts.rcp_d == 0.0f || s != e4m3_from_f32(__fmul_rn(q, 1.0f + 0x1p-21f)))
      s = e4m3_from_f32(__fdiv_rn(amax_blk, ts.d));
  }
  *st = scale_step(s, ts);
  return s;
}

// ------------------------------------------------------------------ block encode by table
// The streaming encoders take a block's bracket from a per-CTA table indexed by the
// scale byte (256 entries per tensor scale g, built once per CTA), leave the rare
// elements where the bracket straddles a threshold to a per-lane fix-up after the
// whole iteration, and keep the common path free of branches.
//
// The bracket (rlo, rhi) of 1/t for the decode step t of one scale byte:
//   t == 0       -> (0, 0): every product is a signed zero, which is the code of a
//                   block with t == 0;
//   certifiable  -> the verified bracket of block_step;
//   otherwise    -> (0, +inf): the two codes of every nonzero element differ (zero
//                   and a saturated or NaN product), so each goes to e2m1_fix.
__device__ __forceinline__ float2 step_bracket(float t) {
  if (!(t > 0.0f)) return make_float2(0.0f, 0.0f);
  const BlockStep b = block_step(t);
  return step_certifiable(b) ? make_float2(b.rlo, b.rhi)
                             : make_float2(0.0f, __int_as_float(0x7F800000));
}

// Entry s of the bracket table of a tensor scale g.
__device__ __forceinline__ float2 bracket_entry(uint32_t s, float g) {
  return step_bracket(__fmul_rn(e4m3_to_f32(s), g));
}

// The block scale byte e4m3(RN(amax_blk / d)): from the product with RN(1/d) when
// both ends of its error interval (as in block_scale_fast) round to the same byte,
// which one conversion of the pair decides; otherwise from the division.
__device__ __forceinline__ uint32_t scale_byte(float amax_blk, const TensorScale& ts) {
  const float q = __fmul_rn(amax_blk, ts.rcp_d);
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
      : "=h"(r)
      : "f"(__fmul_rn(q, 1.0f + 0x1p-21f)), "f"(__fmul_rn(q, 1.0f - 0x1p-21f)));
  const uint32_t lo = r & 0xFFu;
  if (lo == (uint32_t)(r >> 8) && ts.rcp_d > 0.0f) return lo;
  return ts.g == 0.0f ? 0u : e4m3_from_f32(__fdiv_rn(amax_blk, ts.d));
}

// The 16 codes of one block (w0: elements 0..7, w1: 8..15, element i in bits 4i..4i+3)
// from the products with rlo, and the nibbles where the products with rhi disagree.
__device__ __forceinline__ void codes16(const float* f, float2 br, uint32_t& w0, uint32_t& w1,
                                        uint32_t& d0, uint32_t& d1) {
  w0 = e2m1x8_of_products(f, br.x);
  w1 = e2m1x8_of_products(f + 8, br.x);
  d0 = w0 ^ e2m1x8_of_products(f, br.y);
  d1 = w1 ^ e2m1x8_of_products(f + 8, br.y);
}

// The exact code of x under step t where the bracket's codes lo (from rlo) and hi
// (from rhi) differ.  Adjacent magnitudes of one sign leave one threshold m between
// them, decided as in fix_straddles; anything else comes from a block whose products
// are not certified and takes the full exact decision.
__device__ __forceinline__ uint32_t e2m1_fix(float x, float t, uint32_t lo, uint32_t hi) {
  const uint32_t c = lo & 7u;
  if (((lo ^ hi) & 8u) == 0u && (hi & 7u) == c + 1u) {
    const float2 dv = e2m1x2_to_f32x2(c | ((c + 1u) << 4));
    const float m = __fmul_rn(__fadd_rn(dv.x, dv.y), 0.5f);
    const float hh = __int_as_float((__float_as_int(m) & 0x7F800000) - (24 << 23));
    const float hl = c == 0u ? __fmul_rn(hh, 0.5f) : hh;
    const float D = __fmaf_rn(-m, t, fabsf(x));
    const uint32_t mag =
        D > __fmul_rn(hh, t) ? c + 1u : (D >= -__fmul_rn(hl, t) ? c + (c & 1u) : c);
    return (sign_bit(x) << 3) | mag;
  }
  return e2m1_code_exact(x, t);
}

// Codes w with the nibbles flagged in d replaced by e2m1_fix; elem(i) gives the value
// of element i (0..7) of the word.  Visits only the flagged elements.
template <class Elem>
__device__ __forceinline__ uint32_t fix_word(uint32_t w, uint32_t d, float t, Elem elem) {
#pragma unroll 1
  while (d) {
    const uint32_t sh = ((uint32_t)__ffs(d) - 1u) & ~3u;  // 4 i
    const uint32_t dn = (d >> sh) & 0xFu;
    d ^= dn << sh;
    const uint32_t lo = (w >> sh) & 0xFu;
    const uint32_t c = e2m1_fix(elem(sh >> 2), t, lo, lo ^ dn);
    w ^= (lo ^ c) << sh;
  }
  return w;
}

// Element i (runtime, 0..7) of eight packed BF16 values, as FP32.
__device__ __forceinline__ float bf16x8_at(const uint4& v, uint32_t i) {
  const uint32_t h = i >> 1;
  const uint32_t w = h == 0 ? v.x : (h == 1 ? v.y : (h == 2 ? v.z : v.w));
  return __uint_as_float((i & 1u) ? (w & 0xFFFF0000u) : (w << 16));
}

// max(|a|, |b|) of two BF16 pairs, lane by lane; the sign bits are garbage (the xor of
// the inputs') and masked by the caller.  Finite inputs: a NaN would lose.
__device__ __forceinline__ uint32_t maxabs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// max |x| over 16 BF16 values (two 16-byte vectors) as FP32 bits: seven packed
// max-abs operations, then the larger of the two halves.
__device__ __forceinline__ uint32_t absmax_bf16x16_bits(const uint4& a, const uint4& b) {
  PACT_NAN_BF16X2(a.x), PACT_NAN_BF16X2(a.y), PACT_NAN_BF16X2(a.z), PACT_NAN_BF16X2(a.w);
  PACT_NAN_BF16X2(b.x), PACT_NAN_BF16X2(b.y), PACT_NAN_BF16X2(b.z), PACT_NAN_BF16X2(b.w);
  const uint32_t m =
      maxabs_bf16x2(maxabs_bf16x2(maxabs_bf16x2(a.x, a.y), maxabs_bf16x2(a.z, a.w)),
                    maxabs_bf16x2(maxabs_bf16x2(b.x, b.y), maxabs_bf16x2(b.z, b.w))) &
      0x7FFF7FFFu;
  return max(m << 16, m & 0xFFFF0000u);
}

// Offset of the scale word of blocks 4 cg .. 4 cg + 3 of row r (the 128x4 atom layout
// of sf_offset; upr = blocks per row / 4).  32-bit: callers keep pad128(M) * K / 16
// below 2^31.
__device__ __forceinline__ uint32_t sf_word_offset(uint32_t r, uint32_t cg, uint32_t upr) {
  return ((r >> 7) * upr + cg) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u;
}

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// An E4M3 byte -> FP16 (exact: E4M3 values are FP16 normals), in both halves.
__device__ __forceinline__ __half2 e4m3_dup_h2(uint32_t b) {
  uint32_t h2;
  const uint16_t in = (uint16_t)((b & 0xFFu) * 0x0101u);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return *reinterpret_cast<__half2*>(&h2);
}

// Two E2M1 codes (the low byte of `byte`, first element in the low nibble) times
// a block scale -> BF16x2, exactly: the codes convert exactly to FP16, the product
// of an E2M1 value and an E4M3 scale has at most 6 significant bits and lies in
// [2^-10, 2688] (or is zero), so the FP16 multiply, the widening to FP32 and the
// narrowing to BF16 are all exact.  Register-only (no lookup table).
__device__ __forceinline__ uint32_t e2m1x2_scaled_bf16x2(uint32_t byte, __half2 s) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  const float2 f = __half22float2(__hmul2(*reinterpret_cast<__half2*>(&h2), s));
  return pack_bf16x2(f.x, f.y);
}

// max |bf16| over 8 packed values, as FP32 bits (non-negative, so unsigned order).
__device__ __forceinline__ uint32_t absmax_bf16x8_bits(const uint4& v) {
  PACT_NAN_BF16X2(v.x), PACT_NAN_BF16X2(v.y), PACT_NAN_BF16X2(v.z), PACT_NAN_BF16X2(v.w);
  uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                        __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  uint32_t hi = m >> 16, lo = m & 0xFFFFu;
  return (hi > lo ? hi : lo) << 16;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// A read-only 16-byte load that allocates in L1: for a lane that reads a contiguous
// run in several loads, the later loads of a 32-byte sector hit L1.
__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Block-wide max of non-negative float bits, folded into *dst with one atomic per CTA.
__device__ __forceinline__ void block_max_atomic(uint32_t v, unsigned* dst) {
  __shared__ uint32_t red[32];
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int nw = (blockDim.x + 31) >> 5;
    uint32_t x = lane < nw ? red[lane] : 0u;
    x = __reduce_max_sync(0xFFFFFFFFu, x);
    if (lane == 0 && x != 0u) atomicMax(dst, x);
  }
  __syncthreads();  // red[] may be reused by a following call
}

// ------------------------------------------------------------------ exp recipe
// exp(x) by a fixed FP32 recipe (Cody-Waite reduction with a 16-bit head of ln 2,
// degree-7 Taylor polynomial in Horner form with fused multiply-adds, exact
// scaling by 2^n), so that independent implementations agree bit for bit.
__device__ __forceinline__ float scale_pow2(float p, int n) {
  if (n > 127) return __fmul_rn(__fmul_rn(p, 0x1p+64f), __int_as_float((n - 64 + 127) << 23));
  if (n < -126) return __fmul_rn(__fmul_rn(p, __int_as_float((n + 64 + 127) << 23)), 0x1p-64f);
  return __fmul_rn(p, __int_as_float((n + 127) << 23));
}

__device__ __forceinline__ float pexp(float x) {
  if (x != x) return x;
  if (x > 0x1.62e42ep+6f) return __int_as_float(0x7F800000);
  if (x < -0x1.9fe368p+6f) return 0.0f;
  float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float f = __fmaf_rn(-n, 0x1.62e400p-1f, x);
  f = __fmaf_rn(-n, 0x1.7f7d1cp-20f, f);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, f, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, f, 0x1.111112p-7f);
  p = __fmaf_rn(p, f, 0x1.555556p-5f);
  p = __fmaf_rn(p, f, 0x1.555556p-3f);
  p = __fmaf_rn(p, f, 0x1.000000p-1f);
  p = __fmaf_rn(p, f, 1.0f);
  p = __fmaf_rn(p, f, 1.0f);
  return scale_pow2(p, (int)n);
}

// pexp for |x| <= 87: the same operations without the range checks (n stays in
// [-126, 126], so 2^n is a normal number and the final product is exact or
// correctly rounded exactly as in pexp).
__device__ __forceinline__ float pexp_mid(float x) {
  float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float f = __fmaf_rn(-n, 0x1.62e400p-1f, x);
  f = __fmaf_rn(-n, 0x1.7f7d1cp-20f, f);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, f, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, f, 0x1.111112p-7f);
  p = __fmaf_rn(p, f, 0x1.555556p-5f);
  p = __fmaf_rn(p, f, 0x1.555556p-3f);
  p = __fmaf_rn(p, f, 0x1.000000p-1f);
  p = __fmaf_rn(p, f, 1.0f);
  p = __fmaf_rn(p, f, 1.0f);
  return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// h = (g / (1 + exp(-g))) * u, FP32, fixed order.
__device__ __forceinline__ float silu_mul(float g, float u) {
  float e = fabsf(g) <= 87.0f ? pexp_mid(-g) : pexp(-g);
  float den = __fadd_rn(1.0f, e);
  float s = __fdiv_rn(g, den);
  return __fmul_rn(s, u);
}

// A fast stand-in for silu_mul, used only to decide where the exact value is
// needed: h ~ g * u / (1 + e) with e = 2^y, y = -g log2(e), from the hardware
// base-2 exponential and reciprocal (flush-to-zero forms).  The rounding error of
// y (up to 115.5 * 2^-24 for |g| <= 80) is split off with a fused multiply-add
// (together with the low part of log2(e)) and applied to the exponential as
// e (1 + dy ln 2), so what remains is the two approximations (about 2^-22 and
// 2^-23), four roundings and silu_mul's own distance to the true value (about 4
// units): below 2^-20.5 relative for finite inputs with |g| zero or in [2^-60, 80]
// and a normal result (every intermediate is normal there: 1 + e <= 2^116 and
// |g| / (1 + e) >= 2^-110).  kSiluRel keeps a margin of more than 5 over that.
// A subnormal h may flush to a zero of the same sign.
constexpr float kSiluRel = 0x1p-18f;
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  const float ng = -g;
  const float y = __fmul_rn(ng, 0x1.715476p+0f);                            // RN(-g log2 e)
  const float dy = __fmaf_rn(ng, 0x1.4ae0c0p-26f, __fmaf_rn(ng, 0x1.715476p+0f, -y));
  const float e0 = ex2_ftz(y);
  const float e = __fmaf_rn(e0, __fmul_rn(dy, 0x1.62e430p-1f), e0);          // e0 (1 + dy ln 2)
  return __fmul_rn(__fmul_rn(g, rcp_ftz(__fadd_rn(1.0f, e))), u);
}

// silu_mul_fast for two elements at once: the same operations with packed FP32
// pairs (each lane rounds exactly as the scalar operation does), so each result
// is bit-identical to silu_mul_fast; the two MUFU steps stay scalar.
__device__ __forceinline__ float2 silu_mul_fast2(float2 g, float2 u) {
  const float2 ng = make_float2(-g.x, -g.y);
  const float2 l2e = make_float2(0x1.715476p+0f, 0x1.715476p+0f);
  const float2 y = __fmul2_rn(ng, l2e);
  const float2 dy = __ffma2_rn(ng, make_float2(0x1.4ae0c0p-26f, 0x1.4ae0c0p-26f),
                               __ffma2_rn(ng, l2e, make_float2(-y.x, -y.y)));
  const float2 e0 = make_float2(ex2_ftz(y.x), ex2_ftz(y.y));
  const float2 e =
      __ffma2_rn(e0, __fmul2_rn(dy, make_float2(0x1.62e430p-1f, 0x1.62e430p-1f)), e0);
  const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), e);
  return __fmul2_rn(__fmul2_rn(g, make_float2(rcp_ftz(d.x), rcp_ftz(d.y))), u);
}

}  // namespace pact
