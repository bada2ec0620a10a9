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

// Prep: the small adapter layouts the two kernels below and the fused GEMM read.
//   fwd:   At [RP, K] = A^T zero padded (the down-projection's B fragments become
//          single 8-byte loads), Bt [N, RP] = B^T zero padded (GEMM right operand)
//   dgrad: Ap [K, RP] = A zero padded (GEMM right operand)
// One thread per output row; reads are coalesced along the long dimension.
template <int RP>
__global__ void __launch_bounds__(256) k_lora_prep(const uint16_t* __restrict__ A,
                                                   const uint16_t* __restrict__ B, int r,
                                                   int64_t K, int64_t N, int fwd,
                                                   uint16_t* __restrict__ at_out,
                                                   uint16_t* __restrict__ rhs_out) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (fwd) {
    if (t < N) {  // Bt row n
      uint16_t v[RP];
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = j < r ? B[(int64_t)j * N + t] : (uint16_t)0;
      store_row<RP>(rhs_out + t * RP, v);
    } else if (t < N + K) {  // At column k: element (j, k) for every j
      const int64_t k = t - N;
#pragma unroll 4
      for (int j = 0; j < RP; ++j) at_out[(int64_t)j * K + k] = j < r ? A[k * r + j] : (uint16_t)0;
    }
  } else if (t < K) {  // Ap row k
    uint16_t v[RP];
#pragma unroll
    for (int j = 0; j < RP; ++j) v[j] = j < r ? A[t * r + j] : (uint16_t)0;
    store_row<RP>(rhs_out + t * RP, v);
  }
}

// T' = f * (X~ A): x_codes [M, K/2], x_sf (128x4 atoms), At [RP, K].  A CTA owns 16
// rows; warp w takes the 64-wide K chunks w, w+8, ... with two chunks of codes in
// flight ahead of the one it multiplies.  E2M1 pairs are decoded through a
// 256-entry byte -> BF16x2 table in shared memory and scaled by the block's E4M3
// scale with one exact BF16x2 multiply.
template <int RP>
__global__ void __launch_bounds__(256) k_lora_down_fwd(const uint8_t* __restrict__ xc,
                                                       const uint8_t* __restrict__ xsf,
                                                       const float* __restrict__ gx,
                                                       const float* __restrict__ gw, int64_t M,
                                                       int64_t K, const uint16_t* __restrict__ At,
                                                       int r, float scale,
                                                       uint16_t* __restrict__ t_out) {
  constexpr int NT = RP / 8;
  __shared__ float red[8 * 16 * RP];
  __shared__ uint32_t dec[256];
  {
    const float2 f = e2m1x2_to_f32x2(threadIdx.x);
    dec[threadIdx.x] = pack_bf16x2(f.x, f.y);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.x * 16;
  const int64_t ra = m0 + g, rb = m0 + g + 8;
  const bool va = ra < M, vb = rb < M;
  const int64_t c16p = K >> 4;
  float acc[NT][4];
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) acc[jn][0] = acc[jn][1] = acc[jn][2] = acc[jn][3] = 0.0f;

  struct Chunk {
    uint2 qa, qb;
    uint32_t sa, sb;
  };
  // chunk ch of 64 along K: lane (g, c) holds block 4ch + c of rows g and g+8
  auto load = [&](int64_t ch, Chunk& q) {
    const int64_t blk = ch * 4 + c;
    q.qa = q.qb = make_uint2(0, 0);
    q.sa = q.sb = 0;
    if (va) {
      q.qa = __ldg(reinterpret_cast<const uint2*>(xc + ra * (K >> 1) + blk * 8));
      q.sa = xsf[sf_offset(ra, blk, c16p)];
    }
    if (vb) {
      q.qb = __ldg(reinterpret_cast<const uint2*>(xc + rb * (K >> 1) + blk * 8));
      q.sb = xsf[sf_offset(rb, blk, c16p)];
    }
  };
  const int64_t nchunks = K >> 6;
  Chunk q0, q1;
  if (warp < nchunks) load(warp, q0);
  if (warp + 8 < nchunks) load(warp + 8, q1);
  for (int64_t ch = warp; ch < nchunks; ch += 8) {
    Chunk q2;
    if (ch + 16 < nchunks) load(ch + 16, q2);  // two chunks ahead
    const __nv_bfloat162 sca = __float2bfloat162_rn(e4m3_to_f32(q0.sa));
    const __nv_bfloat162 scb = __float2bfloat162_rn(e4m3_to_f32(q0.sb));
    const int64_t kbase = (ch * 4 + c) * 16;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint32_t wa = (s < 2 ? q0.qa.x : q0.qa.y) >> (16 * (s & 1));
      const uint32_t wb = (s < 2 ? q0.qb.x : q0.qb.y) >> (16 * (s & 1));
      uint32_t a[4];
      __nv_bfloat162 t;
      t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&dec[wa & 0xFFu]), sca);
      a[0] = *reinterpret_cast<uint32_t*>(&t);  // row g,   k 4s, 4s+1
      t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&dec[wb & 0xFFu]), scb);
      a[1] = *reinterpret_cast<uint32_t*>(&t);  // row g+8, k 4s, 4s+1
      t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&dec[(wa >> 8) & 0xFFu]), sca);
      a[2] = *reinterpret_cast<uint32_t*>(&t);  // row g,   k 4s+2, 4s+3
      t = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&dec[(wb >> 8) & 0xFFu]), scb);
      a[3] = *reinterpret_cast<uint32_t*>(&t);  // row g+8, k 4s+2, 4s+3
      const int64_t k = kbase + 4 * s;
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        // At rows >= r are zero, so no bounds test on the adapter column is needed
        const uint2 bb = __ldg(reinterpret_cast<const uint2*>(At + (int64_t)(jn * 8 + g) * K + k));
        const uint32_t b[2] = {bb.x, bb.y};
        mma_bf16_16816(acc[jn], a, b);
      }
    }
    q0 = q1;
    q1 = q2;
  }
  const float ga = *gx, gb = *gw;
  const bool normal = __fmul_rn(ga, gb) > 0.0f;
  const float f = normal ? __fdiv_rn(scale, gb) : __fmul_rn(scale, ga);
  reduce_and_store<RP>(acc, red, m0, M, f, t_out);
}

// U' = f * (dY B^T): dy [M, N] BF16, B [r, N] row-major.  A CTA owns 16 rows; warp
// w takes the 64-wide N chunks w, w+8, ... with two chunks in flight ahead.
template <int RP>
__global__ void __launch_bounds__(256) k_lora_down_dgrad(const uint16_t* __restrict__ dy,
                                                         const float* __restrict__ gdy,
                                                         const float* __restrict__ gw,
                                                         int64_t M, int64_t N,
                                                         const uint16_t* __restrict__ B, int r,
                                                         float scale,
                                                         uint16_t* __restrict__ u_out) {
  constexpr int NT = RP / 8;
  __shared__ float red[8 * 16 * RP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.x * 16;
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
  uint4 x0[4], x1[4];
  if (warp < nchunks) load(warp, x0);
  if (warp + 8 < nchunks) load(warp + 8, x1);
  for (int64_t ch = warp; ch < nchunks; ch += 8) {
    uint4 x2[4];
    if (ch + 16 < nchunks) load(ch + 16, x2);  // two chunks ahead
    const int64_t n0 = ch * 64 + 16 * c;
    const uint32_t wa[8] = {x0[0].x, x0[0].y, x0[0].z, x0[0].w, x0[1].x, x0[1].y, x0[1].z, x0[1].w};
    const uint32_t wb[8] = {x0[2].x, x0[2].y, x0[2].z, x0[2].w, x0[3].x, x0[3].y, x0[3].z, x0[3].w};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4] = {wa[2 * s], wb[2 * s], wa[2 * s + 1], wb[2 * s + 1]};
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const int col = jn * 8 + g;
        uint32_t b[2] = {0u, 0u};
        if (col < r) {
          const uint2 bb = __ldg(reinterpret_cast<const uint2*>(B + (int64_t)col * N + n0 + 4 * s));
          b[0] = bb.x;
          b[1] = bb.y;
        }
        mma_bf16_16816(acc[jn], a, b);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x0[i] = x1[i];
      x1[i] = x2[i];
    }
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
                          uint16_t* bt_out, uint16_t* at_ws, cudaStream_t stream) {
  note_launch();
  k_lora_prep<RP><<<(int)((N + K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 1, at_ws,
                                                                    bt_out);
  note_launch();
  k_lora_down_fwd<RP><<<(int)((M + 15) / 16), 256, 0, stream>>>(xc, xsf, gx, gw, M, K, at_ws, r,
                                                                 scale, t_out);
  return cudaGetLastError();
}

template <int RP>
static cudaError_t dgrad_rp(const uint16_t* dy, const float* gdy, const float* gw, int64_t M,
                            int64_t N, const uint16_t* A, const uint16_t* B, int r, float scale,
                            int64_t K, uint16_t* u_out, uint16_t* ap_out, cudaStream_t stream) {
  note_launch();
  k_lora_prep<RP><<<(int)((K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 0, nullptr, ap_out);
  note_launch();
  k_lora_down_dgrad<RP><<<(int)((M + 15) / 16), 256, 0, stream>>>(dy, gdy, gw, M, N, B, r, scale,
                                                                   u_out);
  return cudaGetLastError();
}

cudaError_t launch_lora_down_fwd(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                 const float* gw, int64_t M, int64_t K, const uint16_t* A,
                                 const uint16_t* B, int r, int rp, float scale, int64_t N,
                                 uint16_t* t_out, uint16_t* bt_out, uint16_t* at_ws,
                                 cudaStream_t stream) {
  if (rp == 16)
    return fwd_rp<16>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, at_ws,
                      stream);
  if (rp == 32)
    return fwd_rp<32>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, at_ws,
                      stream);
  return fwd_rp<64>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, t_out, bt_out, at_ws, stream);
}

cudaError_t launch_lora_down_dgrad(const uint16_t* dy, const float* gdy, const float* gw,
                                   int64_t M, int64_t N, const uint16_t* A, const uint16_t* B,
                                   int r, int rp, float scale, int64_t K, uint16_t* u_out,
                                   uint16_t* ap_out, cudaStream_t stream) {
  if (rp == 16) return dgrad_rp<16>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
  if (rp == 32) return dgrad_rp<32>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
  return dgrad_rp<64>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
}

}  // namespace pact
