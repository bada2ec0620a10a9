// LoRA down-projections feeding the fused NVFP4 GEMM.
//
// "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 7 "LoRA branch":
// BF16 GEMMs on the reconstructed (dequantised) shared NVFP4 input in the
// forward; BF16 input gradients in the backward.  Figure 3: the adapter output is
// added to the frozen projection's output.
//
//   forward:  T = Xhat A        Xhat = dequant(Xq) [M, K], A [K, r]   -> [M, r]
//   dgrad:    U = dY B^T        dY BF16 [M, N],    B [r, N]           -> [M, r]
//
// The result v = f * T is stored as BF16 [M, 2 RP] (RP = r rounded up to 16, 32 or
// 64, zero padded): columns [0, RP) hold hi = bf16(v) and [RP, 2 RP) hold
// lo = bf16(v - hi); the GEMM multiplies both halves by the same right operand
// ([N, RP] = B^T or [K, RP] = A, zero padded), so the fused BF16 LoRA product
// hi B + lo B carries v to about 16 bits
// (a single BF16 rounding of v costs up to 2^-9 |v| |B| per term, more than the
// output tolerance allows).  f is chosen so that the GEMM epilogue's single
// scale s = g_a g_w turns the fused product into the LoRA term:
//   forward  f = scale / g_w       (s T' B = g_x g_w X~ A B scale / g_w = scale Xhat A B)
//   dgrad    f = scale / (g_dy g_w)
// and f = scale * g_x (forward) or scale (dgrad) when g_a g_w == 0 (the epilogue
// then uses s = 1 and the NVFP4 operand is all zero).  Here X~ = e2m1 * e4m3 is
// the dequantised input without g, which BF16 holds exactly.
//
// These GEMMs are skinny (r <= 64) and bound by reading Xq or dY once, so they run
// on BF16 mma.sync (m16n8k16, FP32 accumulate) fed straight from registers.  A
// CTA owns 16 rows; its 8 warps split K in 64-wide chunks and reduce through
// shared memory.  Inside a chunk, lane (g, c) holds block c (16 elements) of rows
// g and g+8; the MMA's k index is permuted accordingly on both operands.
#include "common.cuh"
#include "kernels.h"

namespace pact {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Two E2M1 codes (one byte) times an E4M3 scale -> BF16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_scaled_bf16x2(uint32_t byte, __half2 sc) {
  uint32_t h2;
  uint16_t in = (uint16_t)(byte & 0xFFu);
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "h"(in));
  __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h2), sc);
  float2 f = __half22float2(v);
  return pack_bf16x2(f.x, f.y);
}

// Sums the 8 warps' partial products and stores f * T as a BF16 pair per element:
// out[m, j] = hi = bf16(v), out[m, RP + j] = lo = bf16(v - hi), so that the fused
// GEMM's BF16 LoRA product sees v to about 16 significant bits.
template <int RP>
__device__ __forceinline__ void reduce_and_store(float (*acc)[4], float* red, int64_t m0,
                                                 int64_t M, float f, uint16_t* out) {
  constexpr int NT = RP / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // red[warp][row 0..15][col 0..RP)
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) {
    float* r0 = red + (warp * 16 + g) * RP + jn * 8 + 2 * c;
    float* r1 = red + (warp * 16 + g + 8) * RP + jn * 8 + 2 * c;
    r0[0] = acc[jn][0];
    r0[1] = acc[jn][1];
    r1[0] = acc[jn][2];
    r1[1] = acc[jn][3];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 16 * RP; e += blockDim.x) {
    const int row = e / RP, col = e - row * RP;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[(w * 16 + row) * RP + col];
    const int64_t m = m0 + row;
    if (m < M) {
      const float v = s * f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      out[m * (2 * RP) + col] = *reinterpret_cast<const uint16_t*>(&hi);
      out[m * (2 * RP) + RP + col] = *reinterpret_cast<const uint16_t*>(&lo);
    }
  }
}

// One padded right-operand row for the fused GEMM: the row's r adapter values,
// zero padded to RP (the GEMM multiplies it by both halves of the left operand).
template <int RP>
__device__ __forceinline__ void store_row(uint16_t* out_row, const uint16_t* v) {
  uint4* o = reinterpret_cast<uint4*>(out_row);
#pragma unroll
  for (int i = 0; i < RP / 8; ++i)
    o[i] = make_uint4((uint32_t)v[8 * i] | ((uint32_t)v[8 * i + 1] << 16),
                      (uint32_t)v[8 * i + 2] | ((uint32_t)v[8 * i + 3] << 16),
                      (uint32_t)v[8 * i + 4] | ((uint32_t)v[8 * i + 5] << 16),
                      (uint32_t)v[8 * i + 6] | ((uint32_t)v[8 * i + 7] << 16));
}

// T' = f * (X~ A): x_codes [M, K/2], x_sf (128x4 atoms), A [K, r] row-major.
// The first tcta CTAs write Bt [N, RP] = B^T zero padded (one row per thread, reads of
// B coalesced along N); the rest own 16 rows of X each.
template <int RP>
__global__ void __launch_bounds__(256) k_lora_down_fwd(const uint8_t* __restrict__ xc,
                                                       const uint8_t* __restrict__ xsf,
                                                       const float* __restrict__ gx,
                                                       const float* __restrict__ gw, int64_t M,
                                                       int64_t K, const uint16_t* __restrict__ A,
                                                       const uint16_t* __restrict__ B, int r,
                                                       float scale, int64_t N,
                                                       uint16_t* __restrict__ t_out,
                                                       uint16_t* __restrict__ bt_out, int tcta) {
  constexpr int NT = RP / 8;
  __shared__ float red[8 * 16 * RP];
  if ((int)blockIdx.x < tcta) {
    const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n < N) {
      uint16_t v[RP];
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = j < r ? B[(int64_t)j * N + n] : (uint16_t)0;
      store_row<RP>(bt_out + n * RP, v);
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t m0 = (int64_t)(blockIdx.x - tcta) * 16;
  const int64_t ra = m0 + g, rb = m0 + g + 8;
  const bool va = ra < M, vb = rb < M;
  const int64_t c16p = K >> 4;
  float acc[NT][4];
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) acc[jn][0] = acc[jn][1] = acc[jn][2] = acc[jn][3] = 0.0f;

  // chunk ch of 64 along K: lane (g, c) holds block 4ch + c of rows g and g+8
  auto load = [&](int64_t ch, uint2& qa, uint2& qb, uint32_t& sa, uint32_t& sb) {
    const int64_t blk = ch * 4 + c;
    qa = make_uint2(0, 0);
    qb = make_uint2(0, 0);
    sa = sb = 0;
    if (va) {
      qa = *reinterpret_cast<const uint2*>(xc + ra * (K >> 1) + blk * 8);
      sa = xsf[sf_offset(ra, blk, c16p)];
    }
    if (vb) {
      qb = *reinterpret_cast<const uint2*>(xc + rb * (K >> 1) + blk * 8);
      sb = xsf[sf_offset(rb, blk, c16p)];
    }
  };
  const int64_t nchunks = K >> 6;
  uint2 qa, qb;
  uint32_t sa, sb;
  if (warp < nchunks) load(warp, qa, qb, sa, sb);
  for (int64_t ch = warp; ch < nchunks; ch += 8) {
    uint2 nqa, nqb;
    uint32_t nsa, nsb;
    if (ch + 8 < nchunks) load(ch + 8, nqa, nqb, nsa, nsb);  // prefetch the next chunk
    const __half2 sca = __half2half2(__float2half_rn(e4m3_to_f32(sa)));
    const __half2 scb = __half2half2(__float2half_rn(e4m3_to_f32(sb)));
    const int64_t kbase = (ch * 4 + c) * 16;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t wa = (s < 2 ? qa.x : qa.y) >> (16 * (s & 1));
      const uint32_t wb = (s < 2 ? qb.x : qb.y) >> (16 * (s & 1));
      uint32_t a[4];
      a[0] = e2m1x2_scaled_bf16x2(wa & 0xFFu, sca);         // row g,   k 4s, 4s+1
      a[1] = e2m1x2_scaled_bf16x2(wb & 0xFFu, scb);         // row g+8, k 4s, 4s+1
      a[2] = e2m1x2_scaled_bf16x2((wa >> 8) & 0xFFu, sca);  // row g,   k 4s+2, 4s+3
      a[3] = e2m1x2_scaled_bf16x2((wb >> 8) & 0xFFu, scb);  // row g+8, k 4s+2, 4s+3
      const int64_t k = kbase + 4 * s;
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const int col = jn * 8 + g;
        uint32_t b[2] = {0u, 0u};
        if (col < r) {
          const uint16_t* ap = A + k * r + col;
          b[0] = (uint32_t)ap[0] | ((uint32_t)ap[r] << 16);
          b[1] = (uint32_t)ap[2 * r] | ((uint32_t)ap[3 * r] << 16);
        }
        mma_bf16_16816(acc[jn], a, b);
      }
    }
    qa = nqa;
    qb = nqb;
    sa = nsa;
    sb = nsb;
  }
  const float ga = *gx, gb = *gw;
  const bool normal = __fmul_rn(ga, gb) > 0.0f;
  const float f = normal ? __fdiv_rn(scale, gb) : __fmul_rn(scale, ga);
  reduce_and_store<RP>(acc, red, m0, M, f, t_out);
}

// U' = f * (dY B^T): dy [M, N] BF16, B [r, N] row-major.
// The first tcta CTAs write Ap [K, RP] = A zero padded; the rest own 16 rows of dY each.
template <int RP>
__global__ void __launch_bounds__(256) k_lora_down_dgrad(const uint16_t* __restrict__ dy,
                                                         const float* __restrict__ gdy,
                                                         const float* __restrict__ gw,
                                                         int64_t M, int64_t N,
                                                         const uint16_t* __restrict__ A,
                                                         const uint16_t* __restrict__ B, int r,
                                                         float scale, int64_t K,
                                                         uint16_t* __restrict__ u_out,
                                                         uint16_t* __restrict__ ap_out, int tcta) {
  constexpr int NT = RP / 8;
  __shared__ float red[8 * 16 * RP];
  if ((int)blockIdx.x < tcta) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < K) {
      uint16_t v[RP];
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = j < r ? A[k * r + j] : (uint16_t)0;
      store_row<RP>(ap_out + k * RP, v);
    }
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t m0 = (int64_t)(blockIdx.x - tcta) * 16;
  const int64_t ra = m0 + g, rb = m0 + g + 8;
  const bool va = ra < M, vb = rb < M;
  float acc[NT][4];
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) acc[jn][0] = acc[jn][1] = acc[jn][2] = acc[jn][3] = 0.0f;

  // chunk ch of 64 along N: lane (g, c) holds elements 16c .. 16c+15 of rows g, g+8
  auto load = [&](int64_t ch, uint4* x) {
    const int64_t n0 = ch * 64 + 16 * c;
    x[0] = x[1] = x[2] = x[3] = make_uint4(0, 0, 0, 0);
    if (va) {
      const uint4* p = reinterpret_cast<const uint4*>(dy + ra * N + n0);
      x[0] = ldg_stream(p);
      x[1] = ldg_stream(p + 1);
    }
    if (vb) {
      const uint4* p = reinterpret_cast<const uint4*>(dy + rb * N + n0);
      x[2] = ldg_stream(p);
      x[3] = ldg_stream(p + 1);
    }
  };
  const int64_t nchunks = N >> 6;
  uint4 x[4];
  if (warp < nchunks) load(warp, x);
  for (int64_t ch = warp; ch < nchunks; ch += 8) {
    uint4 nx[4];
    if (ch + 8 < nchunks) load(ch + 8, nx);  // prefetch the next chunk
    const int64_t n0 = ch * 64 + 16 * c;
    const uint32_t wa[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
    const uint32_t wb[8] = {x[2].x, x[2].y, x[2].z, x[2].w, x[3].x, x[3].y, x[3].z, x[3].w};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4] = {wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1]};
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const int col = jn * 8 + g;
        uint32_t b[2] = {0u, 0u};
        if (col < r) {
          const uint2 bb = *reinterpret_cast<const uint2*>(B + (int64_t)col * N + n0 + 4 * s);
          b[0] = bb.x;
          b[1] = bb.y;
        }
        mma_bf16_16816(acc[jn], a, b);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = nx[i];
  }
  const float ga = *gdy, gb = *gw;
  const float s_main = __fmul_rn(ga, gb);
  const float f = s_main > 0.0f ? __fdiv_rn(scale, s_main) : scale;
  reduce_and_store<RP>(acc, red, m0, M, f, u_out);
}

template <int RP>
static cudaError_t fwd_rp(const uint8_t* xc, const uint8_t* xsf, const float* gx,
                          const float* gw, int64_t M, int64_t K, const uint16_t* A,
                          const uint16_t* B, int r, float scale, int64_t N, uint16_t* t_out,
                          uint16_t* bt_out, int, cudaStream_t stream) {
  const int row_ctas = (int)((M + 15) / 16);
  const int tcta = (int)((N + 255) / 256);
  note_launch();
  k_lora_down_fwd<RP><<<tcta + row_ctas, 256, 0, stream>>>(xc, xsf, gx, gw, M, K, A, B, r,
                                                           scale, N, t_out, bt_out, tcta);
  return cudaGetLastError();
}

template <int RP>
static cudaError_t dgrad_rp(const uint16_t* dy, const float* gdy, const float* gw, int64_t M,
                            int64_t N, const uint16_t* A, const uint16_t* B, int r, float scale,
                            int64_t K, uint16_t* u_out, uint16_t* ap_out, int,
                            cudaStream_t stream) {
  const int row_ctas = (int)((M + 15) / 16);
  const int tcta = (int)((K + 255) / 256);
  note_launch();
  k_lora_down_dgrad<RP><<<tcta + row_ctas, 256, 0, stream>>>(dy, gdy, gw, M, N, A, B, r, scale,
                                                             K, u_out, ap_out, tcta);
  return cudaGetLastError();
}

cudaError_t launch_lora_down_fwd(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                 const float* gw, int64_t M, int64_t K, const uint16_t* A,
                                 const uint16_t* B, int r, int rp, float scale, int64_t N,
                                 uint16_t* t_out, uint16_t* bt_out, int num_sms,
                                 cudaStream_t stream) {
  if (rp == 16)
    return fwd_rp<16>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, num_sms,
                      stream);
  if (rp == 32)
    return fwd_rp<32>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, num_sms,
                      stream);
  return fwd_rp<64>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, num_sms,
                    stream);
}

cudaError_t launch_lora_down_dgrad(const uint16_t* dy, const float* gdy, const float* gw,
                                   int64_t M, int64_t N, const uint16_t* A, const uint16_t* B,
                                   int r, int rp, float scale, int64_t K, uint16_t* u_out,
                                   uint16_t* ap_out, int num_sms, cudaStream_t stream) {
  if (rp == 16)
    return dgrad_rp<16>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, num_sms, stream);
  if (rp == 32)
    return dgrad_rp<32>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, num_sms, stream);
  return dgrad_rp<64>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, num_sms, stream);
}

}  // namespace pact
