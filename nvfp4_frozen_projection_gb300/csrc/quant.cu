// Activation quantisation and frozen-weight packing to NVFP4.
//
// "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs", Table 6 (format) and
// Table 7 (NVFP4 GEMM operands; cached forward and backward weight layouts).
//
// Both operations are HBM-bound and two-pass: the per-tensor scale g = amax/2688
// must be known before the first code is written, so pass 1 reduces amax into a
// device word and pass 2 re-reads the tensor (mostly from L2) and encodes it.
#include "common.cuh"
#include "encode_tiles.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

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
    PACT_NAN_F32(__uint_as_float(a.x)), PACT_NAN_F32(__uint_as_float(a.y));
    PACT_NAN_F32(__uint_as_float(a.z)), PACT_NAN_F32(__uint_as_float(a.w));
    m = max(m, max(max(a.x & 0x7FFFFFFFu, a.y & 0x7FFFFFFFu),
                   max(a.z & 0x7FFFFFFFu, a.w & 0x7FFFFFFFu)));
  }
  block_max_atomic(m, amax_bits);
}

// ---------------------------------------------------------------- pass 2: encode
// The BF16 values themselves, through the shared tile encoder (encode_tiles.cuh).
struct QuantValues {
  __device__ __forceinline__ void row(uint32_t) {}
  __device__ __forceinline__ uint32_t block(const uint4& a, const uint4& b, uint32_t, float* f) {
    bf16x8_to_f32(a, f);
    bf16x8_to_f32(b, f + 8);
    return absmax_bf16x16_bits(a, b);
  }
  __device__ __forceinline__ float elem(const uint4& a, uint32_t i, uint32_t) {
    return bf16x8_at(a, i);
  }
};

__global__ void __launch_bounds__(kTileThreads, 2) k_quant_bf16(
    const __grid_constant__ CUtensorMap tmx, int64_t M, int64_t K, int64_t Mpad, FastDiv upr_div,
    const float* __restrict__ amax_opt, const unsigned* __restrict__ amax_bits,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ g_out,
    unsigned* __restrict__ status) {
  extern __shared__ uint8_t qsm[];
  const TensorScale ts = tensor_scale(amax_opt ? *amax_opt : __uint_as_float(*amax_bits));
  if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = ts.g;
  QuantValues op;
  encode_tiles(&tmx, M, K, Mpad, upr_div, ts, codes, sf, status, qsm, op);
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

cudaError_t launch_quant_bf16(const CUtensorMap& tmx, const uint16_t* x, int64_t M, int64_t K,
                              int64_t ldx, const float* amax_opt, uint8_t* codes, uint8_t* sf,
                              float* g, unsigned* ws_amax, unsigned* status, int num_sms,
                              cudaStream_t stream) {
  if (!amax_opt) {
    cudaError_t e = cudaMemsetAsync(ws_amax, 0, sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    note_launch();
    k_amax_bf16<<<grid_for(M * K / 8, 256, num_sms * 4), 256, 0, stream>>>(x, M, K, ldx,
                                                                            ws_amax);
  }
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        k_quant_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tile_encode_smem_bytes());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t Mpad = pad_to(M, 128);
  const int64_t ntiles = (Mpad / 32) * (K / 64);
  note_launch();
  k_quant_bf16<<<grid_for(ntiles, kTileWarps, num_sms * 2), kTileThreads,
                 tile_encode_smem_bytes(), stream>>>(tmx, M, K, Mpad,
                                                     FastDiv::make((uint32_t)(K / 64)), amax_opt,
                                                     ws_amax, codes, sf, g, status);
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
