/*
 * Plain CPU oracle for the NVFP4 LoRA-linear hot path.  TEST INFRASTRUCTURE ONLY:
 * it is called by tests/, by the smoke check and by the CPU-baseline leg of the
 * benchmark, never by the product library.  It shares no code with the CUDA path.
 *
 * Source: "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs"
 *   - Table 6 (NVFP4 format parameters): E2M1 elements, one E4M3 scale per
 *     16-element block, 4.5 bits per element.
 *   - Table 7 (precision allocation): activations and the frozen weight are NVFP4,
 *     RMSNorm normalises in FP32 and keeps an FP32 per-token statistic,
 *     SiLU-multiply computes in FP32 and keeps separate gate/up copies.
 *   - The abstract: cached forward and backward weight layouts.
 * The pages fix neither the per-tensor scale nor the operation order; this file
 * takes the plain readings listed beside each function (all are repeated, with
 * their reasons, in the design notes of the repository).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * Every FP32 expression below is one IEEE operation rounded to nearest-even;
 * -ffp-contract=off keeps the compiler from fusing a multiply and an add.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- E2M1 / E4M3 */

/* The eight E2M1 magnitudes (1 sign, 2 exponent, 1 mantissa bit; Table 6). */
static const float kE2M1Mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float orc_e2m1_decode(uint32_t code) {
  float m = kE2M1Mag[code & 7u];
  return (code & 8u) ? -m : m;
}

/* E4M3 ("fn" variant: bias 7, no infinities, 0x7F/0xFF are NaN, max 448). */
float orc_e4m3_decode(uint32_t byte) {
  uint32_t b = byte & 0xFFu;
  uint32_t s = b >> 7, e = (b >> 3) & 15u, m = b & 7u;
  float v;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    v = ldexpf((float)m, -9);                 /* subnormal: (m/8) * 2^-6 */
  else
    v = ldexpf((float)(8u + m), (int)e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Round |v| to the nearest E2M1 magnitude, ties to the even code, saturating at 6.
 * The code's sign bit is the sign bit of v, so negative values that round to zero
 * give the code 0x8 (negative zero). */
uint32_t orc_e2m1_encode(float v) {
  uint32_t sign = signbit(v) ? 8u : 0u;
  float a = fabsf(v);
  uint32_t idx = 0;
  for (uint32_t i = 0; i < 7; ++i) {
    float mid = 0.5f * (kE2M1Mag[i] + kE2M1Mag[i + 1]); /* exact in FP32 */
    if (a < mid) { idx = i; break; }
    if (a == mid) { idx = (i % 2u == 0u) ? i : i + 1u; break; }
    idx = i + 1u;
  }
  return sign | idx;
}

/* Round a non-negative v to E4M3 (nearest, ties to even, subnormals included) and
 * saturate to the finite maximum 448 (code 0x7E). */
uint32_t orc_e4m3_encode(float v) {
  if (!(v > 0.0f)) return 0u;
  if (v >= 448.0f) return 0x7Eu;
  int e2;
  (void)frexpf(v, &e2);
  int E = e2 - 1;                         /* v in [2^E, 2^(E+1)) */
  if (E < -6) {                           /* subnormal grid, step 2^-9 */
    float q = rintf(ldexpf(v, 9));        /* exact scaling, then RNE */
    return (uint32_t)q;                   /* q == 8 is the smallest normal, code 0x08 */
  }
  int q = (int)rintf(ldexpf(v, 3 - E));   /* significand * 8, in [8, 16] */
  if (q == 16) { q = 8; E += 1; }
  uint32_t code = ((uint32_t)(E + 7) << 3) | (uint32_t)(q - 8);
  return code > 0x7Eu ? 0x7Eu : code;
}

/* ------------------------------------------------------- per-tensor FP32 scale */

/* amax_t = max |x|, exact. */
float orc_amax(const float* x, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = fabsf(x[i]);
    if (v > a) a = v;
  }
  return a;
}

/* g = amax_t / (6 * 448): the per-tensor scale chosen so that the largest block
 * scale is exactly the E4M3 maximum.  6*448 = 2688 is exact, so this is one RN
 * division. */
float orc_global_scale(float amax) { return amax / 2688.0f; }

/* Encode one block of 16 values that share the E4M3 scale s (already chosen).
 * t = e4m3(s) * g is the block's decode step (one FP32 product), and each element
 * is divided by it, one IEEE division rounded to nearest:
 *   q = e2m1(x / t),
 * the element formula q = e2m1_rne_sat(x / (s g)) with its FP32 order written out.
 * If t is zero (a zero block, a zero tensor, or an underflowed product) every code
 * is a signed zero.  A quotient that overflows saturates to 6. */
static void encode_block(const float* x, int64_t stride, float t, uint32_t* codes16) {
  for (int i = 0; i < 16; ++i) {
    float v = x[(int64_t)i * stride];
    if (t == 0.0f)
      codes16[i] = signbit(v) ? 8u : 0u;
    else
      codes16[i] = orc_e2m1_encode(v / t);
  }
}

/* Block scale for a block whose absolute maximum is amax_blk:
 *   d = 6 * g;  s = e4m3(amax_blk / d).   A zero g gives s = 0. */
static uint32_t block_scale(float amax_blk, float g) {
  if (g == 0.0f) return 0u;
  float d = 6.0f * g;
  return orc_e4m3_encode(amax_blk / d);
}

static void put_nibble(uint8_t* codes, int64_t row_bytes, int64_t r, int64_t c, uint32_t q) {
  uint8_t* p = codes + r * row_bytes + c / 2;
  if ((c & 1) == 0)
    *p = (uint8_t)((*p & 0xF0u) | (q & 0xFu));       /* even column: low nibble */
  else
    *p = (uint8_t)((*p & 0x0Fu) | ((q & 0xFu) << 4)); /* odd column: high nibble */
}

/* Quantise the rows of x [R, C] (row stride ldx, C % 16 == 0) with 1x16 blocks
 * along each row, given the per-tensor scale g.
 * codes: [R, C/2] bytes, two E2M1 codes per byte, even column in the low nibble.
 * scales: [R, C/16] E4M3 bytes in logical (row-major) order. */
void orc_quant_rows(const float* x, int64_t R, int64_t C, int64_t ldx, float g,
                    uint8_t* codes, uint8_t* scales) {
  int64_t nb = C / 16;
  memset(codes, 0, (size_t)(R * (C / 2)));
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = x + r * ldx + b * 16;
      float amax_blk = 0.0f;
      for (int i = 0; i < 16; ++i) {
        float v = fabsf(blk[i]);
        if (v > amax_blk) amax_blk = v;
      }
      uint32_t s = block_scale(amax_blk, g);
      float t = orc_e4m3_decode(s) * g;
      uint32_t q[16];
      encode_block(blk, 1, t, q);
      for (int i = 0; i < 16; ++i) put_nibble(codes, C / 2, r, b * 16 + i, q[i]);
      scales[r * nb + b] = (uint8_t)s;
    }
  }
}

/* Frozen-weight pack (cached forward and backward layouts, abstract and Table 7).
 * W is [N, K] (Y = X W^T).  One E4M3 scale per 16x16 tile of W, so that the
 * forward layout (blocks of 16 along K) and the backward layout (blocks of 16
 * along N) hold the same effective weights: dequant(bwd) == dequant(fwd)^T.
 * codes_fwd [N, K/2], sf_fwd [N, K/16]; codes_bwd [K, N/2], sf_bwd [K, N/16]
 * (scales in logical row-major order).  N % 16 == 0 and K % 16 == 0. */
void orc_pack_weight(const float* W, int64_t N, int64_t K, float g,
                     uint8_t* codes_fwd, uint8_t* sf_fwd,
                     uint8_t* codes_bwd, uint8_t* sf_bwd) {
  memset(codes_fwd, 0, (size_t)(N * (K / 2)));
  memset(codes_bwd, 0, (size_t)(K * (N / 2)));
  for (int64_t tn = 0; tn < N / 16; ++tn) {
    for (int64_t tk = 0; tk < K / 16; ++tk) {
      float amax_tile = 0.0f;
      for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j) {
          float v = fabsf(W[(tn * 16 + i) * K + tk * 16 + j]);
          if (v > amax_tile) amax_tile = v;
        }
      uint32_t s = block_scale(amax_tile, g);
      float t = orc_e4m3_decode(s) * g;
      for (int i = 0; i < 16; ++i) {
        int64_t n = tn * 16 + i;
        uint32_t q[16];
        encode_block(W + n * K + tk * 16, 1, t, q);
        for (int j = 0; j < 16; ++j) {
          int64_t k = tk * 16 + j;
          put_nibble(codes_fwd, K / 2, n, k, q[j]);
          put_nibble(codes_bwd, N / 2, k, n, q[j]);
        }
        sf_fwd[n * (K / 16) + tk] = (uint8_t)s;
      }
      for (int j = 0; j < 16; ++j) sf_bwd[(tk * 16 + j) * (N / 16) + tn] = (uint8_t)s;
    }
  }
}

/* Exact dequantisation x = e2m1(q) * e4m3(s) * g, in FP64 (at most 6 significant
 * bits times the 24 of g, so no rounding happens). */
void orc_dequant_rows(const uint8_t* codes, const uint8_t* scales, float g,
                      int64_t R, int64_t C, double* out) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) {
      uint8_t byte = codes[r * (C / 2) + c / 2];
      uint32_t q = (c & 1) ? (byte >> 4) : (byte & 0xFu);
      double s = (double)orc_e4m3_decode(scales[r * (C / 16) + c / 16]);
      out[r * C + c] = (double)orc_e2m1_decode(q) * s * (double)g;
    }
}

/* -------------------------------------------------------------------- RMSNorm */

/* RMSNorm forward statistic and FP32 output (Table 7: BF16 input, FP32
 * normalisation, FP32 per-token statistic kept for backward).  The FP32 sum of
 * squares is order dependent, so the order is fixed: the row is split into
 * blocks of 16; virtual lane l (0..31) takes blocks l, l+32, l+64, ... in
 * increasing order and adds x_i*x_i one element at a time; the 32 partial sums
 * are then combined by a butterfly (offsets 16, 8, 4, 2, 1), which leaves the
 * same total in every lane.
 *   ms = ss / H;  rstd = 1 / sqrt(ms + eps);  y_j = (x_j * rstd) * gamma_j.
 * x: [R, H] (BF16 values widened to FP32), gamma: [H], H % 16 == 0. */
void orc_rmsnorm_rows(const float* x, const float* gamma, int64_t R, int64_t H, float eps,
                      float* rstd, float* y) {
  int64_t nb = H / 16;
  for (int64_t r = 0; r < R; ++r) {
    const float* xr = x + r * H;
    float acc[32];
    for (int l = 0; l < 32; ++l) {
      float a = 0.0f;
      for (int64_t b = l; b < nb; b += 32)
        for (int i = 0; i < 16; ++i) {
          float v = xr[b * 16 + i];
          float sq = v * v;
          a = a + sq;
        }
      acc[l] = a;
    }
    for (int off = 16; off >= 1; off >>= 1) {
      float nxt[32];
      for (int l = 0; l < 32; ++l) nxt[l] = acc[l] + acc[l ^ off];
      memcpy(acc, nxt, sizeof(acc));
    }
    float ss = acc[0];
    float ms = ss / (float)H;
    float den = sqrtf(ms + eps);
    float rs = 1.0f / den;
    rstd[r] = rs;
    for (int64_t j = 0; j < H; ++j) {
      float n = xr[j] * rs;
      y[r * H + j] = n * gamma[j];
    }
  }
}

/* ------------------------------------------------------------ exp and SiLU */

/* exp(x) in FP32 by a fixed recipe, so that two implementations of the recipe
 * give identical bits (the C library's expf and a GPU's may differ in the last
 * place).  Method: Cody and Waite's argument reduction x = n*ln2 + f with ln2
 * split into a 16-bit head and a tail (so n*ln2_hi is exact), the degree-7
 * Taylor polynomial of e^f evaluated by Horner's rule with fused multiply-adds,
 * and an exact scaling by 2^n.  Overflow above the largest x whose exponential
 * is finite; zero below ln(2^-150). */
#define PEXP_HI   0x1.62e42ep+6f    /* largest float with exp(x) < FLT_MAX */
#define PEXP_LO  -0x1.9fe368p+6f    /* ~ ln(2^-150) */
#define PEXP_L2E  0x1.715476p+0f    /* log2(e) rounded to FP32 */
#define PEXP_LN2H 0x1.62e400p-1f    /* head of ln 2 (16 significant bits) */
#define PEXP_LN2L 0x1.7f7d1cp-20f   /* ln 2 - head, rounded to FP32 */

float orc_pexp(float x) {
  if (x != x) return x;
  if (x > PEXP_HI) return INFINITY;
  if (x < PEXP_LO) return 0.0f;
  float n = rintf(x * PEXP_L2E);
  float f = fmaf(-n, PEXP_LN2H, x);
  f = fmaf(-n, PEXP_LN2L, f);
  /* Taylor coefficients 1/k!, k = 7 .. 0, each rounded to FP32 */
  float p = 0x1.a01a02p-13f;
  p = fmaf(p, f, 0x1.6c16c2p-10f);
  p = fmaf(p, f, 0x1.111112p-7f);
  p = fmaf(p, f, 0x1.555556p-5f);
  p = fmaf(p, f, 0x1.555556p-3f);
  p = fmaf(p, f, 0x1.000000p-1f);
  p = fmaf(p, f, 1.0f);
  p = fmaf(p, f, 1.0f);
  return ldexpf(p, (int)n); /* exact, or correctly rounded when subnormal */
}

/* SiLU-multiply forward (Table 7: BF16 gate/up inputs, FP32 arithmetic):
 *   e = exp(-gate);  h = (gate / (1 + e)) * up. */
void orc_silu_mul(const float* gate, const float* up, int64_t n, float* h) {
  for (int64_t i = 0; i < n; ++i) {
    float e = orc_pexp(-gate[i]);
    float den = 1.0f + e;
    float s = gate[i] / den;
    h[i] = s * up[i];
  }
}

/* Row-strided variant for a fused [M, 2I] gate|up tensor. */
void orc_silu_mul_rows(const float* gateup, int64_t M, int64_t I, float* h) {
  for (int64_t r = 0; r < M; ++r)
    orc_silu_mul(gateup + r * 2 * I, gateup + r * 2 * I + I, I, h + r * I);
}

/* Element-wise pexp over an array (test convenience). */
void orc_pexp_array(const float* x, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_pexp(x[i]);
}

/* Element-wise codecs over arrays (test convenience). */
void orc_e2m1_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(v[i]);
}
void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(v[i]);
}
