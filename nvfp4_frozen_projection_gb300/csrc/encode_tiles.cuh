// Streaming NVFP4 encode of a row-major [M, K] tensor read as BF16 through TMA tiles
// (the activation quantiser and the RMSNorm -> NVFP4 encode share it; they differ in
// the FP32 value each element is encoded from).
//
// Tile = 32 rows x 64 columns (4 KB), lane = one row of it: a unit of four
// consecutive blocks (128 bytes).  Each warp runs its own two-stage ring: its lane 0
// fetches the warp's next tiles by TMA (128-byte swizzle, so that each lane's reads
// of its own row are free of bank conflicts), and the warp encodes one tile while
// the next is in flight.  Warps take tiles in turn over the tensor, tile t covering
// row group t / (K/64) and column group t % (K/64), so the warps of the grid sweep
// the tensor front to back.  A unit's four scale bytes are one 4-byte word of the
// 128x4 atom layout (K/16 is a multiple of 4), stored whole; its 32 code bytes leave
// as two 16-byte stores.  The brackets come from the CTA's table (bracket_entry);
// elements where a bracket straddles a threshold (about one in 10^3) are fixed after
// the unit's four blocks are encoded, from the values still held in registers.
// Rows past M read as zeros (the tensor map's bounds) and store zero scale words up
// to pad128(M), so the padded scale array is fully defined.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pact {

constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileStages = 2;
constexpr uint32_t kTileBytes = 32 * 128;
constexpr uint64_t kTileWaitNs = 2000000000ull;

// Dynamic shared memory of a kernel that calls encode_tiles (1 KB alignment slack).
// Kernels run two CTAs of 256 threads per SM: with three, the 80-register cap made
// the encode spill and both encoders ran 8-14 % slower (measured on GB300).
inline size_t tile_encode_smem_bytes() {
  return 1024 + (size_t)kTileWarps * kTileStages * kTileBytes;
}

// The encode loop.  Called by every thread of a CTA of kTileThreads threads.  tmx:
// BF16 map over the input, box 64 x 32, 128-byte swizzle.  Op supplies the values:
//   op.row(r)                  per tile, for the lane's row r < M;
//   op.block(a, b, col, f)     the 16 FP32 values of the block whose BF16 inputs are
//                              a, b (columns col .. col + 15) into f; returns their
//                              max |.| as FP32 bits;
//   op.elem(a, i, col)         element i of the 8 inputs a (columns col .. col + 7),
//                              the same FP32 value block() gave.
template <class Op>
__device__ __forceinline__ void encode_tiles(const CUtensorMap* tmx, int64_t M, int64_t K,
                                             int64_t Mpad, FastDiv upr_div, const TensorScale& ts,
                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                             unsigned* __restrict__ status, uint8_t* dsm, Op& op) {
  __shared__ float2 brk[256];
  __shared__ __align__(8) uint64_t full[kTileWarps][kTileStages];
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  brk[threadIdx.x] = bracket_entry(threadIdx.x, ts.g);  // blockDim.x == 256
  if (lane == 0) {
    for (int i = 0; i < kTileStages; ++i) mbar_init(smem_addr(&full[warp][i]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t ring = ((smem_addr(dsm) + 1023u) & ~1023u) + warp * kTileStages * kTileBytes;
  const uint32_t upr = (uint32_t)(K >> 6);  // column groups (units per row)
  const uint32_t ntiles = (uint32_t)(Mpad >> 5) * upr;
  const uint32_t sf_bytes = (uint32_t)Mpad * upr * 4u;
  const uint32_t first = blockIdx.x * kTileWarps + warp, step = gridDim.x * kTileWarps;
  auto issue = [&](uint32_t t, int slot) {
    const uint32_t rg = upr_div.div(t), cg = t - rg * upr;
    const uint32_t bar = smem_addr(&full[warp][slot]);
    mbar_expect_tx(bar, kTileBytes);
    tma_load_2d(ring + slot * kTileBytes, tmx, (int32_t)(cg * 64u), (int32_t)(rg * 32u), bar);
  };
  if (lane == 0) {
    prefetch_tensormap(tmx);
    for (int i = 0; i < kTileStages; ++i)
      if (first + i * step < ntiles) issue(first + i * step, i);
  }
  uint32_t k = 0;
  for (uint32_t t = first; t < ntiles; t += step, ++k) {
    const int slot = (int)(k % kTileStages);
    const bool landed =
        mbar_wait(smem_addr(&full[warp][slot]), (k / kTileStages) & 1u, kTileWaitNs, nullptr);
    if (!__all_sync(0xFFFFFFFFu, landed)) {  // the whole warp leaves together
      // give the warp's other copy in flight a bounded chance to land before leaving
      if (lane == 0) {
        atomicOr(status, PACT_DEV_TIMEOUT);
        const uint32_t k2 = k + 1;
        if (t + step < ntiles)
          mbar_wait(smem_addr(&full[warp][k2 % kTileStages]), (k2 / kTileStages) & 1u,
                    kTileWaitNs, nullptr);
      }
      __syncwarp();
      break;
    }
    const uint32_t row_smem = ring + slot * kTileBytes + lane * 128u;
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = ld_shared_v4(row_smem + ((c ^ (lane & 7u)) << 4));
    __syncwarp();  // every lane's reads of the slot are done
    if (lane == 0 && t + kTileStages * step < ntiles) {
      fence_proxy_async_smem();
      issue(t + kTileStages * step, slot);
    }
    const uint32_t rg = upr_div.div(t), cg = t - rg * upr;
    const uint32_t r = rg * 32u + lane;
    const uint32_t so = sf_word_offset(r, cg, upr);
    if (r >= (uint32_t)M) {
      if (PACT_IN(so + 4u <= sf_bytes)) *reinterpret_cast<uint32_t*>(sf + so) = 0u;
      continue;
    }
    op.row(r);
    const uint32_t col0 = cg * 64u;
    uint32_t w[8], d[8], sw = 0u, any = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float f[16];
      const uint32_t am = op.block(v[2 * j], v[2 * j + 1], col0 + 16u * j, f);
      const uint32_t sb = scale_byte(__uint_as_float(am), ts);
      sw |= sb << (8 * j);
      codes16(f, brk[sb], w[2 * j], w[2 * j + 1], d[2 * j], d[2 * j + 1]);
      any |= d[2 * j] | d[2 * j + 1];
    }
    if (any) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (d[q]) {
          const float tq = __fmul_rn(e4m3_to_f32((sw >> (8 * (q >> 1))) & 0xFFu), ts.g);
          w[q] = fix_word(w[q], d[q], tq,
                          [&](uint32_t i) { return op.elem(v[q], i, col0 + 8u * q); });
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(codes + (int64_t)r * (K >> 1) + cg * 32u);
    if (PACT_IN(cg < upr)) {
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (PACT_IN(so + 4u <= sf_bytes)) *reinterpret_cast<uint32_t*>(sf + so) = sw;
  }
}

}  // namespace pact
