// Activation quantisation and frozen-weight packing to NVFP4.
//
// "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 6 (format) and
// Table 7 (NVFP4 GEMM operands; cached forward and backward weight layouts).
//
// Both operations are HBM-bound and two-pass: the per-tensor scale g = amax/2688
// must be known before the first code is written, so pass 1 reduces amax into a
// device word and pass 2 re-reads the tensor (mostly from L2) and encodes it.
#include "common.cuh"
#include "kernels.h"

namespace pact {

// ---------------------------------------------------------------- pass 1: amax
// max |x| over BF16 [M, K] (row stride ldx elements), folded into *amax_bits.
// Eight 16-byte loads in flight per thread and four CTAs per SM (64 registers):
// 128 KB of reads in flight per SM, what HBM needs at the latency it has under
// full load.
__global__ void __launch_bounds__(256, 4) k_amax_bf16(const uint16_t* __restrict__ x, int64_t M,
                                                      int64_t K, int64_t ldx,
                                                      unsigned* __restrict__ amax_bits) {
  const int64_t vpr = K >> 3;  // 16-byte vectors per row
  const int64_t total = M * vpr;
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (ldx == K) {
    const uint4* p = reinterpret_cast<const uint4*>(x);
    for (; v + 7 * stride < total; v += 8 * stride) {
      uint4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = ldg_stream(p + v + u * stride);
#pragma unroll
      for (int u = 0; u < 8; ++u) m = max(m, absmax_bf16x8_bits(a[u]));
    }
    for (; v < total; v += stride) m = max(m, absmax_bf16x8_bits(ldg_stream(p + v)));
  } else {
    for (; v < total; v += stride) {
      int64_t r = v / vpr, c = v - r * vpr;
      m = max(m, absmax_bf16x8_bits(ldg_stream(x + r * ldx + c * 8)));
    }
  }
  block_max_atomic(m, amax_bits);
}

// max |W| over FP32 [n] (contiguous), folded into *amax_bits.
__global__ void __launch_bounds__(256) k_amax_f32(const float* __restrict__ w, int64_t n,
                                                  unsigned* __restrict__ amax_bits) {
  const int64_t nv = n >> 2;
  uint32_t m = 0;
  const uint4* p = reinterpret_cast<const uint4*>(w);
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nv;
       v += (int64_t)gridDim.x * blockDim.x) {
    uint4 a = ldg_stream(p + v);
    m = max(m, max(max(a.x & 0x7FFFFFFFu, a.y & 0x7FFFFFFFu),
                   max(a.z & 0x7FFFFFFFu, a.w & 0x7FFFFFFFu)));
  }
  block_max_atomic(m, amax_bits);
}

// ---------------------------------------------------------------- pass 2: encode
// Lane = one block of 16 elements, warp = 32 consecutive blocks (a contiguous 1 KB
// of a contiguous tensor), blocks numbered row-major over [pad128(M), K/16].  Each
// lane holds the next block's 32 bytes in flight while it encodes the current one.
// A block's 8 code bytes leave as one 8-byte store (256 contiguous bytes per warp);
// the scale bytes of four consecutive blocks (one 4-byte word of the 128x4 atom
// layout, never split across rows since K/16 is a multiple of 4) are gathered by
// two shuffles and stored by the first lane of the four.  Blocks of rows past M (up
// to pad128(M)) get zero scale bytes so the padded scale array is fully defined.
__device__ __forceinline__ void quant_fetch(const uint16_t* x, int64_t ldx, uint32_t blk,
                                            uint32_t total, uint32_t M, const FastDiv& bpr_div,
                                            uint32_t bpr, uint4& v0, uint4& v1) {
  if (blk < total) {
    const uint32_t r = bpr_div.div(blk);
    if (r < M) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)r * ldx + (blk - r * bpr) * 16);
      v0 = ldg_stream(src);
      v1 = ldg_stream(src + 1);
    }
  }
}

__global__ void __launch_bounds__(256) k_quant_bf16(const uint16_t* __restrict__ x, int64_t M,
                                                    int64_t K, int64_t ldx, int64_t Mpad,
                                                    FastDiv bpr_div,
                                                    const float* __restrict__ amax_opt,
                                                    const unsigned* __restrict__ amax_bits,
                                                    uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ sf,
                                                    float* __restrict__ g_out) {
  const float amax = amax_opt ? *amax_opt : __uint_as_float(*amax_bits);
  const TensorScale ts = tensor_scale(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = ts.g;
  const uint32_t bpr = (uint32_t)(K >> 4);           // blocks per row
  const uint32_t total = (uint32_t)Mpad * bpr;        // < 2^31 (checked by the caller)
  const uint32_t lane = threadIdx.x & 31u;
  // warps take 32-block strips in turn, so each warp iteration covers 1 KB
  const uint32_t stride = gridDim.x * blockDim.x;
  uint32_t blk = blockIdx.x * blockDim.x + threadIdx.x;
  uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
  quant_fetch(x, ldx, blk, total, (uint32_t)M, bpr_div, bpr, n0, n1);
  for (; blk - lane < total; blk += stride) {  // warp-uniform trip count
    const uint4 v0 = n0, v1 = n1;
    quant_fetch(x, ldx, blk + stride, total, (uint32_t)M, bpr_div, bpr, n0, n1);
    const bool live = blk < total;
    const uint32_t r = bpr_div.div(blk), cb = blk - r * bpr;
    uint32_t sb = 0;
    if (live && r < M) {
      float f[16];
      bf16x8_to_f32(v0, f);
      bf16x8_to_f32(v1, f + 8);
      BlockStep st;
      sb = block_scale_fast(__uint_as_float(max(absmax_bf16x8_bits(v0), absmax_bf16x8_bits(v1))),
                            ts, &st);
      const uint2 cw = make_uint2(encode8(f, st), encode8(f + 8, st));
      if (PACT_IN(r < (uint64_t)M && cb < bpr))
        *reinterpret_cast<uint2*>(codes + (int64_t)r * (K >> 1) + cb * 8) = cw;
    }
    // scale bytes of blocks cb .. cb+3 (same row) into one word
    uint32_t w = sb | (__shfl_down_sync(0xFFFFFFFFu, sb, 1) << 8);
    w |= __shfl_down_sync(0xFFFFFFFFu, w, 2) << 16;
    if (live && (cb & 3u) == 0u && PACT_IN(sf_offset(r, cb, bpr) + 4 <= Mpad * (int64_t)bpr))
      *reinterpret_cast<uint32_t*>(sf + sf_offset(r, cb, bpr)) = w;
  }
}

// ---------------------------------------------------------------- weight pack
// One warp per 16x16 tile of W [N, K]: the tile's amax gives one E4M3 scale shared
// by the forward layout ([N, K], blocks along K) and the backward layout ([K, N],
// blocks along N), so both hold the same effective weights.
// Lane l handles tile row l/2, columns 8*(l%2) .. +8.
// gu_half > 0 (forward layout only): the rows are written in the interleaved
// gate|up order (gu_interleaved); 16-row tiles stay whole, so the scales are the
// same bytes, and g is the whole weight's.
__global__ void __launch_bounds__(256) k_pack_weight(const float* __restrict__ W, int64_t N,
                                                     int64_t K,
                                                     const unsigned* __restrict__ amax_bits,
                                                     int backward, int64_t gu_half,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ sf,
                                                     float* __restrict__ g_out) {
  __shared__ uint8_t nib[8][16][17];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TensorScale ts = tensor_scale(__uint_as_float(*amax_bits));
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = ts.g;
  const int64_t tiles_k = K >> 4;
  const int64_t ntiles = (N >> 4) * tiles_k;
  const int i = lane >> 1, h = lane & 1;
  for (int64_t tile = (int64_t)blockIdx.x * 8 + warp; tile < ntiles;
       tile += (int64_t)gridDim.x * 8) {
    const int64_t tn = tile / tiles_k, tk = tile - tn * tiles_k;
    const float4* src = reinterpret_cast<const float4*>(W + (tn * 16 + i) * K + tk * 16 + 8 * h);
    float4 a = __ldg(src), b = __ldg(src + 1);
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, __float_as_uint(f[j]) & 0x7FFFFFFFu);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    BlockStep st;
    const uint32_t s = block_scale(__uint_as_float(m), ts, &st);
    const uint32_t w = encode8(f, st);
    if (!backward) {
      const int64_t n = gu_half ? gu_interleaved(tn * 16 + i, gu_half) : tn * 16 + i;
      if (PACT_IN(n < N && tk < (K >> 4))) {
        *reinterpret_cast<uint32_t*>(codes + n * (K >> 1) + tk * 8 + 4 * h) = w;
        if (h == 0) sf[sf_offset(n, tk, K >> 4)] = (uint8_t)s;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) nib[warp][i][8 * h + j] = (uint8_t)((w >> (4 * j)) & 0xFu);
      __syncwarp();
      // lane now handles backward row k = tk*16 + i, columns n = tn*16 + 8h .. +8
      uint32_t o = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) o |= (uint32_t)nib[warp][8 * h + j][i] << (4 * j);
      const int64_t k = tk * 16 + i;
      if (PACT_IN(k < K && tn < (N >> 4))) {
        *reinterpret_cast<uint32_t*>(codes + k * (N >> 1) + tn * 8 + 4 * h) = o;
        if (h == 0) sf[sf_offset(k, tn, N >> 4)] = (uint8_t)s;
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------- launchers
static int grid_for(int64_t work, int threads, int max_blocks) {
  int64_t b = (work + threads - 1) / threads;
  if (b > max_blocks) b = max_blocks;
  if (b < 1) b = 1;
  return (int)b;
}

cudaError_t launch_amax_bf16(const uint16_t* x, int64_t M, int64_t K, unsigned* ws_amax,
                             int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws_amax, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  note_launch();
  k_amax_bf16<<<grid_for(M * K / 8, 256, num_sms * 4), 256, 0, stream>>>(x, M, K, K, ws_amax);
  return cudaGetLastError();
}

cudaError_t launch_quant_bf16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                              const float* amax_opt, uint8_t* codes, uint8_t* sf, float* g,
                              unsigned* ws_amax, int num_sms, cudaStream_t stream) {
  if (!amax_opt) {
    cudaError_t e = cudaMemsetAsync(ws_amax, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    note_launch();
    k_amax_bf16<<<grid_for(M * K / 8, 256, num_sms * 4), 256, 0, stream>>>(x, M, K, ldx,
                                                                            ws_amax);
  }
  const int64_t Mpad = pad_to(M, 128);
  note_launch();
  k_quant_bf16<<<grid_for(Mpad * (K / 16), 256, num_sms * 8), 256, 0, stream>>>(
      x, M, K, ldx, Mpad, FastDiv::make((uint32_t)(K / 16)), amax_opt, ws_amax, codes, sf, g);
  return cudaGetLastError();
}

cudaError_t launch_pack_weight(const float* W, int64_t N, int64_t K, int backward,
                               int64_t gu_half, uint8_t* codes, uint8_t* sf, float* g,
                               unsigned* ws_amax, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws_amax, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const int64_t rows = backward ? K : N, cols = backward ? N : K;
  e = cudaMemsetAsync(sf, 0, (size_t)(pad_to(rows, 128) * pad_to(cols / 16, 4)), stream);
  if (e != cudaSuccess) return e;
  note_launch();
  k_amax_f32<<<grid_for(N * K / 4, 256, num_sms * 8), 256, 0, stream>>>(W, N * K, ws_amax);
  const int64_t ntiles = (N / 16) * (K / 16);
  note_launch();
  k_pack_weight<<<grid_for(ntiles * 32, 256, num_sms * 16), 256, 0, stream>>>(
      W, N, K, ws_amax, backward, gu_half, codes, sf, g);
  return cudaGetLastError();
}

}  // namespace pact
