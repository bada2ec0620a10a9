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
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pact {

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Sums the 8 warps' partial products (fixed order) and stores f * T as a BF16
// pair per element: out[m, j] = hi = bf16(v), out[m, RP + j] = lo = bf16(v - hi),
// so that the fused GEMM's BF16 LoRA product sees v to about 16 significant bits.
// acc[g][jn][*] is the m16n8 accumulator of row group g (rows 16g + lane/4 and
// 16g + lane/4 + 8) and columns 8 jn + 2 (lane % 4) + {0, 1}.
// Four 8x8 BF16 matrices from shared memory, each transposed: lanes 8i .. 8i + 7
// give the row addresses of matrix i.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// cp.async copies into shared memory; src_bytes = 0 writes zeros instead of reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int RP, int G>
__device__ __forceinline__ void reduce_and_store(float (*acc)[RP / 8][4], float* red, int64_t m0,
                                                 int64_t M, float f, uint16_t* out) {
  constexpr int NT = RP / 8, ROWS = 16 * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // red[warp][row 0..ROWS)[col 0..RP)
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
#pragma unroll
    for (int jn = 0; jn < NT; ++jn) {
      float* r0 = red + (warp * ROWS + 16 * gi + g) * RP + jn * 8 + 2 * c;
      float* r1 = r0 + 8 * RP;
      r0[0] = acc[gi][jn][0];
      r0[1] = acc[gi][jn][1];
      r1[0] = acc[gi][jn][2];
      r1[1] = acc[gi][jn][3];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < ROWS * RP; e += blockDim.x) {
    const int row = e / RP, col = e - row * RP;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[(w * ROWS + row) * RP + col];
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
                                                   int64_t gu_half,
                                                   uint16_t* __restrict__ at_out,
                                                   uint16_t* __restrict__ rhs_out) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (fwd) {
    if (t < N) {  // Bt row n (column gu_logical(n) of B in the interleaved order)
      const int64_t src = gu_half ? gu_logical(t, gu_half) : t;
      uint16_t v[RP];
#pragma unroll
      for (int j = 0; j < RP; ++j) v[j] = j < r ? B[(int64_t)j * N + src] : (uint16_t)0;
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

// Both down-projections are skinny GEMMs ([M, K] x [K, RP]) bound by reading
// their left operand once.  A CTA owns 16 G rows (G = 2 row groups of 16 when
// RP <= 32, else 1); its 8 warps split K into interleaved chunks of 64 bytes per
// row and reduce through shared memory in a fixed order.  Inside a chunk, lane
// (g, c) = (lane / 4, lane % 4) loads 16 contiguous bytes of rows g and g + 8 of
// every row group (a warp instruction covers 8 rows x 64 bytes), and the m16n8k16
// MMAs take the chunk's K elements in a permuted order, the same on both operands:
// step s gives lane c the elements [4s, 4s + 4) of its own 16-byte piece.  The next
// chunk's loads are in flight while the current one is multiplied.

// T' = f * (X~ A): x_codes [M, K/2], x_sf (128x4 atoms), At [RP, K].  A chunk is
// 128 codes of a row: lane c holds blocks 2c and 2c + 1 (32 codes, 16 bytes).  E2M1
// pairs are converted in registers and scaled by their block's E4M3 scale exactly
// (e2m1x2_scaled_bf16x2).
template <int RP, int G>
__global__ void __launch_bounds__(256, 2) k_lora_down_fwd(const uint8_t* __restrict__ xc,
                                                       const uint8_t* __restrict__ xsf,
                                                       const float* __restrict__ gx,
                                                       const float* __restrict__ gw, int64_t M,
                                                       int64_t K, const uint16_t* __restrict__ At,
                                                       float scale, int plain,
                                                       uint16_t* __restrict__ t_out) {
  constexpr int NT = RP / 8;
  __shared__ float red[8 * 16 * G * RP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.x * (16 * G);
  const int64_t c16p = pad_to(K >> 4, 4);
  const int64_t row_bytes = K >> 1;
  const int nch = (int)((K + 127) >> 7);
  // in a final half chunk (K % 128 == 64) lanes 2 and 3 have nothing to load
  const bool half_tail = (K & 127) != 0;
  float acc[G][NT][4];
#pragma unroll
  for (int gi = 0; gi < G; ++gi)
#pragma unroll
    for (int jn = 0; jn < NT; ++jn) acc[gi][jn][0] = acc[gi][jn][1] = acc[gi][jn][2] = acc[gi][jn][3] = 0.0f;

  struct Chunk {
    uint4 q[G][2];      // codes of rows g, g + 8 of each group
    uint32_t sc[G][2];  // the two block scales (2 bytes) of those rows
  };
  auto load = [&](int ch, Chunk& x) {
    const bool live = !(half_tail && ch == nch - 1 && c >= 2);
    const int64_t blk = (int64_t)ch * 8 + 2 * c;  // first of the lane's two blocks
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = m0 + 16 * gi + g + 8 * h;
        x.q[gi][h] = make_uint4(0u, 0u, 0u, 0u);
        x.sc[gi][h] = 0u;
        if (live && r < M) {
          x.q[gi][h] = ldg_stream(reinterpret_cast<const uint4*>(xc + r * row_bytes + blk * 8));
          x.sc[gi][h] = *reinterpret_cast<const uint16_t*>(xsf + sf_offset(r, blk, c16p));
        }
      }
  };
  Chunk x0, x1;
  if (warp < nch) load(warp, x0);
  for (int ch = warp; ch < nch; ch += 8) {
    if (ch + 8 < nch) load(ch + 8, x1);
    const bool live = !(half_tail && ch == nch - 1 && c >= 2);
    __half2 scl[G][2][2];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        scl[gi][h][0] = e4m3_dup_h2(x0.sc[gi][h] & 0xFFu);
        scl[gi][h][1] = e4m3_dup_h2(x0.sc[gi][h] >> 8);
      }
    const int64_t kb = (int64_t)ch * 128 + 32 * c;
    // the chunk's At fragments (lane (g, c): row 8 jn + g, columns kb .. kb + 32),
    // all requested before the first MMA so the chunk pays one L2 round trip
    uint4 bq[NT][4];
#pragma unroll
    for (int jn = 0; jn < NT; ++jn) {
      // At rows >= r are zero; a dead lane of a half chunk multiplies zeros
      const uint4* src = reinterpret_cast<const uint4*>(At + (int64_t)(jn * 8 + g) * K + kb);
#pragma unroll
      for (int i = 0; i < 4; ++i) bq[jn][i] = live ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t bfr[NT][2];
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const uint4 v = bq[jn][s >> 1];
        bfr[jn][0] = (s & 1) ? v.z : v.x;
        bfr[jn][1] = (s & 1) ? v.w : v.y;
      }
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        uint32_t a[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t word = (s < 4 ? (s < 2 ? x0.q[gi][h].x : x0.q[gi][h].y)
                                       : (s < 6 ? x0.q[gi][h].z : x0.q[gi][h].w)) >>
                                (16 * (s & 1));
          a[h] = e2m1x2_scaled_bf16x2(word, scl[gi][h][s >> 2]);            // elements 4s, 4s+1
          a[2 + h] = e2m1x2_scaled_bf16x2(word >> 8, scl[gi][h][s >> 2]);   // elements 4s+2, 4s+3
        }
#pragma unroll
        for (int jn = 0; jn < NT; ++jn) mma_bf16_16816(acc[gi][jn], a, bfr[jn]);
      }
    }
    x0 = x1;
  }
  // plain: f = scale * g_x, i.e. v = scale * (Xhat A) for the adapter gradients
  const float ga = *gx, gb = plain ? 0.0f : *gw;
  const bool normal = !plain && __fmul_rn(ga, gb) > 0.0f;
  const float f = normal ? __fdiv_rn(scale, gb) : __fmul_rn(scale, ga);
  reduce_and_store<RP, G>(acc, red, m0, M, f, t_out);
}

// The NVFP4 quantisation of dY that k_quant_lora_down performs on the way: the
// per-tensor amax (given, or from an amax pass) and the code/scale/g outputs.
struct DyQuant {
  const float* amax_opt;
  const unsigned* amax_bits;
  uint8_t* codes;  // [M, N/2]
  uint8_t* sf;     // 128x4 atoms, rows padded to 128
  float* g_out;
};

// U' = f * (dY B^T), dy [M, N] BF16, B [r, N] row-major, for 128-row blocks of dY
// whose column range is split over a cluster of NS CTAs (NS a power of two <= 8,
// along grid x).  Warp w multiplies rows 16w .. 16w + 15 of the block; the eight
// warps step through the same 64-column chunks, which one thread fetches by TMA into
// a 4-slot ring: per slot the block's 128 dY rows and the chunk of B (r rows), both
// 128-byte rows in the 128-byte swizzle (rows r .. RP - 1 of the B part are zeroed
// once and never copied into).  A slot is refilled when all eight warps have
// released it (an mbarrier with eight arrivals), so warps run ahead of one another
// by up to the ring's depth instead of meeting at a CTA barrier every chunk.  Lane
// (g, c) holds 16
// consecutive elements of rows g and g + 8, [16c, 16c + 16) of the chunk: in K step
// s of the m16n8k16 MMA its k slots 2c, 2c + 1 / 2c + 8, 2c + 9 carry columns
// 16c + 4s + 0, 1 / 2, 3, and the B fragment is read at the same columns (a k
// permutation both operands share).  The CTAs' partial sums meet in distributed
// shared memory at the end: CTA j of the cluster adds the NS partials of rows
// [128 j / NS, 128 (j + 1) / NS) in rank order, so the result does not depend on
// scheduling.
// With QUANT the same pass quantises dY to NVFP4, byte for byte as the quantiser
// does (the same bracket table and element encode): a lane's 16 elements of a row
// are exactly one NVFP4 block.  The grid covers the rows up to the 128-row padding
// of the scale atoms, whose scales encode zero (the rows past M read as zeros).
constexpr int kDyRing = 4;  // chunk slots
constexpr uint64_t kDyWaitNs = 2000000000ull;

template <int RP>
constexpr uint32_t dy_slot_bytes() {
  return 128 * 128 + RP * 128;  // dY rows, then B rows; a multiple of 1024
}
template <int RP>
constexpr int dy_smem_bytes() {
  return 1024 + kDyRing * (int)dy_slot_bytes<RP>();  // >= 128 RP 4 bytes of partial sums
}

// Byte offset of 16-byte chunk q of row `row` in a tile of 128-byte rows written by
// a TMA copy with the 128-byte swizzle (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t q) {
  return row * 128u + ((q ^ (row & 7u)) << 4);
}

template <int RP, bool QUANT>
__global__ void __launch_bounds__(256, 2) k_lora_down_dy(const __grid_constant__ CUtensorMap tm_dy,
                                                         const __grid_constant__ CUtensorMap tm_b,
                                                         const float* __restrict__ gdy,
                                                         const float* __restrict__ gw, int64_t M,
                                                         int64_t N, int r, float scale, int plain,
                                                         uint16_t* __restrict__ u_out, DyQuant qz,
                                                         unsigned* __restrict__ status) {
  constexpr int NT = RP / 8;
  constexpr uint32_t SLOT = dy_slot_bytes<RP>();
  constexpr uint32_t BOFF = 128 * 128;  // B rows follow the dY rows in a slot
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t full[kDyRing], empty[kDyRing];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ns = (int)gridDim.x, split = (int)blockIdx.x;  // split == rank in the cluster
  const int64_t mb0 = (int64_t)blockIdx.y * 128;
  const int nch = (int)(N >> 6);
  const int ch0 = (int)((int64_t)nch * split / ns), ch1 = (int)((int64_t)nch * (split + 1) / ns);
  const uint32_t ring = (smem_addr(dsm) + 1023u) & ~1023u;
  uint8_t* const ring_ptr = dsm + (ring - smem_addr(dsm));
  TensorScale tsq = {0.0f, 0.0f, 0.0f};
  __shared__ float2 brk[QUANT ? 256 : 1];  // bracket table of the dY scale (bracket_entry)
  if constexpr (QUANT) {
    const float amax = qz.amax_opt ? *qz.amax_opt : __uint_as_float(*qz.amax_bits);
    tsq = tensor_scale(amax);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *qz.g_out = tsq.g;
    brk[threadIdx.x] = bracket_entry(threadIdx.x, tsq.g);  // blockDim.x == 256
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDyRing; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), 8);
    }
    fence_mbar_init();
  }
  // rows r .. RP - 1 of every slot's B part stay zero (the copies bring r rows)
  for (int i = threadIdx.x; i < kDyRing * (RP - r) * 32; i += blockDim.x) {
    const int slot = i / ((RP - r) * 32), rem = i - slot * ((RP - r) * 32);
    reinterpret_cast<uint32_t*>(ring_ptr + slot * SLOT + BOFF + r * 128)[rem] = 0u;
  }
  __syncthreads();
  const uint32_t chunk_bytes = BOFF + (uint32_t)r * 128u;
  auto issue = [&](int ch, int slot) {
    const uint32_t bar = smem_addr(&full[slot]);
    mbar_expect_tx(bar, chunk_bytes);
    tma_load_2d(ring + slot * SLOT, &tm_dy, ch * 64, (int32_t)mb0, bar);
    tma_load_2d(ring + slot * SLOT + BOFF, &tm_b, ch * 64, 0, bar);
  };
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tm_dy);
    prefetch_tensormap(&tm_b);
    for (int i = 0; i < kDyRing; ++i)
      if (ch0 + i < ch1) issue(ch0 + i, i);
  }
  const int64_t row0 = mb0 + warp * 16 + g;
  const bool ok0 = row0 < M, ok1 = row0 + 8 < M;
  const uint32_t xr = (uint32_t)(warp * 16 + g);  // tile row of the lane's first row
  float acc[NT][4];
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) acc[jn][0] = acc[jn][1] = acc[jn][2] = acc[jn][3] = 0.0f;
  // scale-byte offsets of the two rows' blocks in chunk 0 (block 4 ch + c of a row
  // sits at ch * 512 + c past them)
  const int64_t c16p = N >> 4;  // N % 64 == 0: no column padding of the scale atoms
  auto sf_row = [&](int64_t row) {
    return ((row >> 7) * (c16p >> 2)) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4 + c;
  };
  const int64_t sfo0 = sf_row(row0), sfo1 = sf_row(row0 + 8);

  for (int cc = ch0; cc < ch1; ++cc) {
    const int k = cc - ch0, slot = k % kDyRing;
    const bool landed =
        mbar_wait(smem_addr(&full[slot]), (uint32_t)(k / kDyRing) & 1u, kDyWaitNs, nullptr);
    if (!__all_sync(0xFFFFFFFFu, landed)) {  // the whole warp leaves together
      if (lane == 0) atomicOr(status, PACT_DEV_TIMEOUT);
      break;
    }
    const uint32_t sb = ring + slot * SLOT;
    uint4 xc[2][2];
    xc[0][0] = ld_shared_v4(sb + swz128(xr, 2 * c));
    xc[0][1] = ld_shared_v4(sb + swz128(xr, 2 * c + 1));
    xc[1][0] = ld_shared_v4(sb + swz128(xr + 8, 2 * c));
    xc[1][1] = ld_shared_v4(sb + swz128(xr + 8, 2 * c + 1));
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint4& lo0 = xc[0][s >> 1];
      const uint4& lo1 = xc[1][s >> 1];
      const uint32_t a[4] = {(s & 1) ? lo0.z : lo0.x, (s & 1) ? lo1.z : lo1.x,
                             (s & 1) ? lo0.w : lo0.y, (s & 1) ? lo1.w : lo1.y};
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const uint32_t brow = (uint32_t)(jn * 8 + g);
        const uint2 bb =
            ld_shared_v2(sb + BOFF + swz128(brow, 2 * c + (s >> 1)) + 8u * (uint32_t)(s & 1));
        const uint32_t bfr[2] = {bb.x, bb.y};
        mma_bf16_16816(acc[jn], a, bfr);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));  // the warp is done with the slot
    // thread 0 refills the slot of the previous chunk once every warp released it
    if (threadIdx.x == 0 && k >= 1 && cc - 1 + kDyRing < ch1) {
      const int ps = (k - 1) % kDyRing;
      if (mbar_wait(smem_addr(&empty[ps]), (uint32_t)((k - 1) / kDyRing) & 1u, kDyWaitNs,
                    nullptr))
        issue(cc - 1 + kDyRing, ps);
      else
        atomicOr(status, PACT_DEV_TIMEOUT);  // the consumers of that chunk time out too
    }
    if constexpr (QUANT) {
      // the lane's two blocks (rows row0 and row0 + 8), brackets from the table; the
      // rare straddling elements are fixed from the registers afterwards
      uint32_t w[4], d[4], sc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        sc[h] = scale_byte(__uint_as_float(absmax_bf16x16_bits(xc[h][0], xc[h][1])), tsq);
        float f[16];
        bf16x8_to_f32(xc[h][0], f);
        bf16x8_to_f32(xc[h][1], f + 8);
        codes16(f, brk[sc[h]], w[2 * h], w[2 * h + 1], d[2 * h], d[2 * h + 1]);
      }
      if (d[0] | d[1] | d[2] | d[3]) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (d[q]) {
            const float tq = __fmul_rn(e4m3_to_f32(sc[q >> 1]), tsq.g);
            w[q] = fix_word(w[q], d[q], tq,
                            [&](uint32_t i) { return bf16x8_at(xc[q >> 1][q & 1], i); });
          }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1];
        const int64_t row = row0 + 8 * h;
        if ((h ? ok1 : ok0) && PACT_IN(row < M && cc < nch))
          *reinterpret_cast<uint2*>(qz.codes + row * (N >> 1) + (int64_t)cc * 32 + 8 * c) =
              make_uint2(w0, w1);
        if (PACT_IN((h ? sfo1 : sfo0) + (int64_t)cc * 512 < pad_to(M, 128) * (N >> 4)))
          qz.sf[(h ? sfo1 : sfo0) + (int64_t)cc * 512] = (uint8_t)sc[h];
      }
    }
  }
  __syncthreads();  // every chunk was consumed: the ring now holds this CTA's partial sums
  float* part = reinterpret_cast<float*>(ring_ptr);  // [128 rows][RP]
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) {
    float* p0 = part + (warp * 16 + g) * RP + jn * 8 + 2 * c;
    *reinterpret_cast<float2*>(p0) = make_float2(acc[jn][0], acc[jn][1]);
    *reinterpret_cast<float2*>(p0 + 8 * RP) = make_float2(acc[jn][2], acc[jn][3]);
  }
  cluster_sync();  // every CTA's partials are in its shared memory
  // plain: f = scale, i.e. v = scale * (dY B^T) for the adapter gradients
  const float s_main = plain ? 0.0f : __fmul_rn(QUANT ? tsq.g : *gdy, *gw);
  const float f = s_main > 0.0f ? __fdiv_rn(scale, s_main) : scale;
  const int rows = 128 / ns;
  for (int e = threadIdx.x; e < rows * RP; e += blockDim.x) {
    const int rl = split * rows + e / RP, col = e % RP;
    const uint32_t local = smem_addr(part + rl * RP + col);
    float sum = 0.0f;
    for (int j = 0; j < ns; ++j) sum += ld_shared_cluster_f32(local, (uint32_t)j);
    const int64_t m = mb0 + rl;
    if (m < M && PACT_IN(col < RP)) {
      const float v = sum * f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      u_out[m * (2 * RP) + col] = *reinterpret_cast<const uint16_t*>(&hi);
      u_out[m * (2 * RP) + RP + col] = *reinterpret_cast<const uint16_t*>(&lo);
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its partials
}

// CTAs per cluster for a dY of N columns: up to 4 while every CTA keeps at least 4
// of the 64-column chunks, and 8 for rows of at least 192 chunks.  Measured on
// GB300 with M = 8192: N = 1024 and 3072 run fastest at 4 (64 row blocks x 4 CTAs
// fill the 152 SMs; 8 CTAs of 6 chunks lose more to each CTA's start-up and cluster
// reduction than they gain), N = 16384 at 8.
static int dy_splits(int64_t N) {
  const int64_t nch = N >> 6;
  int ns = 1;
  while (ns < 4 && 8 * ns <= nch) ns *= 2;
  return nch >= 8 * 24 ? 8 : ns;
}

template <int RP, bool QUANT>
static cudaError_t launch_down_dy(const uint16_t* dy, const float* gdy, const float* gw,
                                  int64_t M, int64_t N, const uint16_t* B, int r, float scale,
                                  int plain, uint16_t* u_out, DyQuant qz, cudaStream_t stream) {
  CUtensorMap tm_dy, tm_b;
  if (make_map(&tm_dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dy, (uint64_t)N, (uint64_t)M, 64, 128,
               CU_TENSOR_MAP_SWIZZLE_128B) ||
      make_map(&tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, (uint64_t)N, (uint64_t)r, 64,
               (uint32_t)r, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  unsigned* status = nullptr;
  cudaError_t e = status_word_ptr(&status);
  if (e != cudaSuccess) return e;
  const int ns = dy_splits(N);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ns, (unsigned)(pad_to(M, 128) / 128));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = dy_smem_bytes<RP>();
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_lora_down_dy<RP, QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dy_smem_bytes<RP>());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, k_lora_down_dy<RP, QUANT>, tm_dy, tm_b, gdy, gw, M, N, r,
                            scale, plain, u_out, qz, status);
}

template <int RP>
static cudaError_t fwd_rp(const uint8_t* xc, const uint8_t* xsf, const float* gx,
                          const float* gw, int64_t M, int64_t K, const uint16_t* A,
                          const uint16_t* B, int r, float scale, int64_t N, int64_t gu_half,
                          uint16_t* t_out, uint16_t* bt_out, uint16_t* at_ws,
                          cudaStream_t stream) {
  constexpr int G = RP <= 32 ? 2 : 1;
  note_launch();
  k_lora_prep<RP><<<(int)((N + K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 1, gu_half,
                                                                    at_ws, bt_out);
  note_launch();
  k_lora_down_fwd<RP, G><<<(int)((M + 16 * G - 1) / (16 * G)), 256, 0, stream>>>(
      xc, xsf, gx, gw, M, K, at_ws, scale, 0, t_out);
  return cudaGetLastError();
}

template <int RP>
static cudaError_t dgrad_rp(const uint16_t* dy, const float* gdy, const float* gw, int64_t M,
                            int64_t N, const uint16_t* A, const uint16_t* B, int r, float scale,
                            int64_t K, uint16_t* u_out, uint16_t* ap_out, cudaStream_t stream) {
  if (ap_out) {  // null: A is already [K, RP] (r == RP) and serves as the GEMM operand
    note_launch();
    k_lora_prep<RP><<<(int)((K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 0, 0, nullptr, ap_out);
  }
  const cudaError_t e = launch_down_dy<RP, false>(dy, gdy, gw, M, N, B, r, scale, 0, u_out,
                                                  DyQuant{}, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_lora_down_fwd(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                 const float* gw, int64_t M, int64_t K, const uint16_t* A,
                                 const uint16_t* B, int r, int rp, float scale, int64_t N,
                                 int64_t gu_half, uint16_t* t_out, uint16_t* bt_out,
                                 uint16_t* at_ws, cudaStream_t stream) {
  if (rp == 16)
    return fwd_rp<16>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, gu_half, t_out, bt_out,
                      at_ws, stream);
  if (rp == 32)
    return fwd_rp<32>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, gu_half, t_out, bt_out,
                      at_ws, stream);
  return fwd_rp<64>(x_codes, x_sf, gx, gw, M, K, A, B, r, scale, N, gu_half, t_out, bt_out,
                    at_ws, stream);
}

cudaError_t launch_lora_down_dgrad(const uint16_t* dy, const float* gdy, const float* gw,
                                   int64_t M, int64_t N, const uint16_t* A, const uint16_t* B,
                                   int r, int rp, float scale, int64_t K, uint16_t* u_out,
                                   uint16_t* ap_out, cudaStream_t stream) {
  if (rp == 16) return dgrad_rp<16>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
  if (rp == 32) return dgrad_rp<32>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
  return dgrad_rp<64>(dy, gdy, gw, M, N, A, B, r, scale, K, u_out, ap_out, stream);
}

template <int RP>
static cudaError_t quant_dgrad_rp(const uint16_t* dy, int64_t M, int64_t N, DyQuant qz,
                                  const float* gw, const uint16_t* A, const uint16_t* B, int r,
                                  float scale, int64_t K, uint16_t* u_out, uint16_t* ap_out,
                                  cudaStream_t stream) {
  if (ap_out) {
    note_launch();
    k_lora_prep<RP><<<(int)((K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 0, 0, nullptr, ap_out);
  }
  const cudaError_t e =
      launch_down_dy<RP, true>(dy, nullptr, gw, M, N, B, r, scale, 0, u_out, qz, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_quant_lora_down(const uint16_t* dy, int64_t M, int64_t N, const float* amax_opt,
                                   unsigned* ws_amax, const float* gw, const uint16_t* A,
                                   const uint16_t* B, int r, int rp, float scale, int64_t K,
                                   uint8_t* codes, uint8_t* sf, float* g, uint16_t* u_out,
                                   uint16_t* ap_out, int num_sms, cudaStream_t stream) {
  if (!amax_opt) {
    cudaError_t e = launch_amax_bf16(dy, M, N, ws_amax, num_sms, stream);
    if (e != cudaSuccess) return e;
  }
  const DyQuant qz{amax_opt, ws_amax, codes, sf, g};
  if (rp == 16) return quant_dgrad_rp<16>(dy, M, N, qz, gw, A, B, r, scale, K, u_out, ap_out, stream);
  if (rp == 32) return quant_dgrad_rp<32>(dy, M, N, qz, gw, A, B, r, scale, K, u_out, ap_out, stream);
  return quant_dgrad_rp<64>(dy, M, N, qz, gw, A, B, r, scale, K, u_out, ap_out, stream);
}

// ============================================================== adapter gradients
// dA = (alpha/r) Xhat^T (dY B^T) [K, r] and dB = (alpha/r) (Xhat A)^T dY [r, N]:
// the down-projection kernels above produce T' = (alpha/r) Xhat A and
// U' = (alpha/r) dY B^T as hi|lo BF16 pairs ("plain" mode), and one tall-skinny
// kernel forms OUT[c, j] = sum_m L[m, c] R[m, j] for L = dY, R = T' (dB) and for
// L = Xhat without its per-tensor scale, R = U' (dA, times g_x afterwards).

// Shared-memory plan of the tall-skinny kernel.  A stage holds ROWS rows of L (the
// 128 columns of the CTA: BF16, or NVFP4 codes plus their 8 block scales) and of R
// (2 RP BF16 columns).  Rows are padded by 16 bytes so that the 8 row addresses of
// a matrix load fall in distinct bank groups.  NVFP4 stages are decoded into one
// BF16 tile before the MMAs read them.
template <int RP, bool FP4>
struct TsPlan {
  static constexpr int ROWS = FP4 ? 64 : 32;
  static constexpr int LST = FP4 ? 64 + 16 : 256 + 16;  // staged L row, bytes
  static constexpr int DST = 256 + 16;                   // decoded BF16 row (NVFP4)
  static constexpr int SFB = FP4 ? 8 : 0;                // block scales per row
  static constexpr int RST = 4 * RP + 16;                // staged R row, bytes
  static constexpr int S_OFF = ROWS * LST;
  static constexpr int R_OFF = S_OFF + ROWS * SFB;
  static constexpr int STAGE = R_OFF + ROWS * RST;
  static constexpr int STAGES = FP4 ? (RP == 64 ? 4 : 6) : 4;
  static constexpr int DEC_OFF = STAGE * STAGES;
  static constexpr int SMEM = DEC_OFF + (FP4 ? ROWS * DST : 0);
};

// OUT partials for 128 columns of L and one split of its rows: OUT[c, j] = sum over
// the split's rows m of L[m, c] R[m, j].  8 warps own 16 columns each.  Every
// thread copies its share of each stage with cp.async (STAGES - 1 stages in flight
// ahead of the one being multiplied; rows past the split read as zeros).
// Transposing matrix loads give the m16n8k16 operands: L^T (16 columns x 16 rows)
// as A and R (16 rows x 8 of its columns, the hi half then the lo half) as B.  The
// split's FP32 sums go to part[split][C][RP] (tr = 0) or part[split][RP][C] (tr = 1),
// the layout whose reduction reads contiguous memory for the final output order.
template <int RP, bool FP4>
__global__ void __launch_bounds__(256, 2) k_lora_ts(const uint16_t* __restrict__ Lb,
                                                    const uint8_t* __restrict__ Lc,
                                                    const uint8_t* __restrict__ Lsf, int64_t M,
                                                    int64_t C, const uint16_t* __restrict__ R,
                                                    int64_t rows_per_split, int tr,
                                                    float* __restrict__ part) {
  using P = TsPlan<RP, FP4>;
  constexpr int NT = RP / 8;
  constexpr int PPR = RP / 4;  // 16-byte pieces per R row
  extern __shared__ __align__(128) uint8_t sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c_base = (int64_t)blockIdx.x * 128;
  const int64_t m_begin = (int64_t)blockIdx.y * rows_per_split;
  const int64_t m_end = min(M, m_begin + rows_per_split);
  const int nr = (int)((m_end - m_begin + P::ROWS - 1) / P::ROWS);
  const int64_t c16p = pad_to(C >> 4, 4);
  const uint32_t sbase = smem_addr(sm);

  auto issue = [&](int i) {
    const uint32_t st = sbase + (uint32_t)((i % P::STAGES) * P::STAGE);
    const int64_t m0 = m_begin + (int64_t)i * P::ROWS;
    if constexpr (FP4) {
      {  // codes: row tid / 4, 16 bytes (32 columns) at piece tid % 4
        const int row = tid >> 2, pc = tid & 3;
        const int64_t m = m0 + row, c = c_base + pc * 32;
        const bool ok = m < m_end && c < C;
        cp_async16(st + row * P::LST + pc * 16, ok ? Lc + m * (C >> 1) + (c >> 1) : Lc, ok ? 16 : 0);
      }
      if (tid < 2 * P::ROWS) {  // scales: row tid / 2, blocks 4h .. 4h + 3 of the tile
        const int row = tid >> 1, h = tid & 1;
        const int64_t m = m0 + row;
        const bool ok = m < m_end && c_base + 64 * h < C;
        cp_async4(st + P::S_OFF + row * 8 + 4 * h,
                  ok ? Lsf + sf_offset(m, (c_base >> 4) + 4 * h, c16p) : Lsf, ok ? 4 : 0);
      }
    } else {
#pragma unroll
      for (int k = 0; k < P::ROWS * 16 / 256; ++k) {  // row p / 16, 8 columns at p % 16
        const int p = tid + 256 * k, row = p >> 4, pc = p & 15;
        const int64_t m = m0 + row, c = c_base + pc * 8;
        const bool ok = m < m_end && c < C;
        cp_async16(st + row * P::LST + pc * 16, ok ? Lb + m * C + c : Lb, ok ? 16 : 0);
      }
    }
    for (int p = tid; p < P::ROWS * PPR; p += 256) {
      const int row = p / PPR, pc = p - row * PPR;
      const int64_t m = m0 + row;
      const bool ok = m < m_end;
      cp_async16(st + P::R_OFF + row * P::RST + pc * 16, ok ? R + m * (2 * RP) + pc * 8 : R,
                 ok ? 16 : 0);
    }
  };

  float acc[NT][4];
#pragma unroll
  for (int jn = 0; jn < NT; ++jn) acc[jn][0] = acc[jn][1] = acc[jn][2] = acc[jn][3] = 0.0f;
#pragma unroll
  for (int s = 0; s < P::STAGES - 1; ++s) {
    if (s < nr) issue(s);
    cp_async_commit();
  }
  for (int i = 0; i < nr; ++i) {
    cp_async_wait<P::STAGES - 2>();
    // stage i has landed for every thread; every thread is done with stage i - 1
    // (and with the decoded tile), so both can be refilled
    __syncthreads();
    if (i + P::STAGES - 1 < nr) issue(i + P::STAGES - 1);
    cp_async_commit();
    const uint8_t* st = sm + (i % P::STAGES) * P::STAGE;
    const uint8_t* Ls = st;
    if constexpr (FP4) {
      // decode: row tid / 4, the 32 columns of piece tid % 4 (blocks 2 pc, 2 pc + 1),
      // exactly: E2M1 x E4M3 products fit in BF16
      const int row = tid >> 2, pc = tid & 3;
      const uint4 q = *reinterpret_cast<const uint4*>(st + row * P::LST + pc * 16);
      const uint32_t sw = *reinterpret_cast<const uint16_t*>(st + P::S_OFF + row * 8 + 2 * pc);
      const __half2 s0 = e4m3_dup_h2(sw & 0xFFu), s1 = e4m3_dup_h2(sw >> 8);
      uint32_t w[16];
#pragma unroll
      for (int b = 0; b < 16; ++b) {
        const uint32_t word = b < 4 ? q.x : (b < 8 ? q.y : (b < 12 ? q.z : q.w));
        w[b] = e2m1x2_scaled_bf16x2(word >> (8 * (b & 3)), b < 8 ? s0 : s1);
      }
      uint4* dst = reinterpret_cast<uint4*>(sm + P::DEC_OFF + row * P::DST + pc * 64);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
      dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
      __syncthreads();
      Ls = sm + P::DEC_OFF;
    }
    constexpr int LS = FP4 ? P::DST : P::LST;
    const uint8_t* Rs = st + P::R_OFF;
#pragma unroll
    for (int ks = 0; ks < P::ROWS / 16; ++ks) {
      uint32_t a[4];
      {
        // matrices: (rows 0-7, cols 0-7), (rows 0-7, cols 8-15), (rows 8-15, cols
        // 0-7), (rows 8-15, cols 8-15) of this k-step and the warp's 16 columns
        const int row = ks * 16 + ((lane >> 4) & 1) * 8 + (lane & 7);
        const int col = warp * 16 + ((lane >> 3) & 1) * 8;
        ldmatrix_x4_trans(a, smem_addr(Ls + row * LS + col * 2));
      }
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        // matrices: rows 0-7 and 8-15 of R columns 8 jn .. (hi), then the same of
        // the lo half (columns RP + 8 jn ..)
        uint32_t b[4];
        const int row = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int col = jn * 8 + ((lane >> 4) & 1) * RP;
        ldmatrix_x4_trans(b, smem_addr(Rs + row * P::RST + col * 2));
        mma_bf16_16816(acc[jn], a, b);
        mma_bf16_16816(acc[jn], a, b + 2);
      }
    }
  }
  cp_async_wait<0>();  // only empty groups can remain; keep the invariant explicit
  // acc[jn]: (column g, j = 8 jn + 2 (lane % 4) + {0, 1}) and (column g + 8, same j)
  const int g = lane >> 2, cq = lane & 3;
  float* out = part + (int64_t)blockIdx.y * C * RP;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t c = c_base + warp * 16 + g + 8 * h;
    if (c < C) {
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) {
        const int j = jn * 8 + 2 * cq;
        if (tr) {
          out[(int64_t)j * C + c] = acc[jn][2 * h];
          out[(int64_t)(j + 1) * C + c] = acc[jn][2 * h + 1];
        } else {
          *reinterpret_cast<float2*>(out + c * RP + j) = make_float2(acc[jn][2 * h], acc[jn][2 * h + 1]);
        }
      }
    }
  }
}

// out = factor * sum over the splits (in split order) of part; layout 0 reads
// part[split][C][RP] and writes out[c * r + j] ([C, r], dA), layout 1 reads
// part[split][RP][C] and writes out[j * C + c] ([r, C], dB).
__global__ void __launch_bounds__(256) k_lora_ts_reduce(const float* __restrict__ part,
                                                        int nsplit, int64_t C, int RP, int r,
                                                        const float* __restrict__ factor,
                                                        int layout, float* __restrict__ out) {
  const float f = factor ? *factor : 1.0f;
  const int64_t total = C * r;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t idx, stride;
    if (layout == 0) {
      const int64_t c = e / r, j = e - c * r;
      idx = c * RP + j;
    } else {
      const int64_t j = e / C, c = e - j * C;
      idx = j * C + c;
    }
    stride = C * RP;
    float s = 0.0f;
    for (int sp = 0; sp < nsplit; ++sp) s += part[(int64_t)sp * stride + idx];
    out[e] = __fmul_rn(s, f);
  }
}

// Row splits of the tall-skinny product.  A fixed model of a 152-SM GPU running two
// CTAs per SM (304 slots) picks the split count: waves of CTAs times the rows each
// streams (plus its partial-sum write), plus the reduction's reads, in units of one
// 128-column row of L.  The plan depends on the shape only, so results are the same
// on every device.
int64_t lora_ts_splits(int64_t M, int64_t C, int rp, bool fp4, int64_t* rows_per_split) {
  const int64_t gran = fp4 ? 64 : 32, slots = 304;
  const double row_bytes = fp4 ? 128 * 0.5625 : 128 * 2.0;
  const double part_rows = 128.0 * rp * 4 / row_bytes;  // one CTA's partial write
  const int64_t ctiles = (C + 127) / 128;
  double best = 1e300;
  int64_t best_ns = 1, best_rps = pad_to(M, gran);
  for (int64_t want = 1; want <= 64; ++want) {
    const int64_t rps = pad_to((M + want - 1) / want, gran);
    const int64_t ns = (M + rps - 1) / rps;
    const int64_t units = ns * ctiles;
    const double cost = (double)((units + slots - 1) / slots) * ((double)rps + part_rows) +
                        (double)units * part_rows / slots;
    if (cost < best - 1e-9) {
      best = cost;
      best_ns = ns;
      best_rps = rps;
    }
  }
  *rows_per_split = best_rps;
  return best_ns;
}

template <int RP, bool FP4>
static cudaError_t launch_ts(const uint16_t* Lb, const uint8_t* Lc, const uint8_t* Lsf, int64_t M,
                             int64_t C, const uint16_t* R, int tr, float* part, int64_t* nsplit,
                             cudaStream_t stream) {
  using P = TsPlan<RP, FP4>;
  static bool attr_set[64] = {};  // per instantiation and device, before its first launch
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(k_lora_ts<RP, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             P::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int64_t rps;
  const int64_t ns = lora_ts_splits(M, C, RP, FP4, &rps);
  *nsplit = ns;
  note_launch();
  k_lora_ts<RP, FP4><<<dim3((unsigned)((C + 127) / 128), (unsigned)ns), 256, P::SMEM, stream>>>(
      Lb, Lc, Lsf, M, C, R, rps, tr, part);
  return cudaSuccess;
}

template <int RP>
static cudaError_t adapter_grad_rp(const uint8_t* xc, const uint8_t* xsf, const float* gx,
                                   int64_t M, int64_t K, const uint16_t* dy, int64_t N,
                                   const uint16_t* A, const uint16_t* B, int r, float scale,
                                   float* dA, float* dB, uint16_t* at_ws, uint16_t* bt_ws,
                                   uint16_t* t_ws, uint16_t* u_ws, float* part, int num_sms,
                                   cudaStream_t stream) {
  constexpr int G = RP <= 32 ? 2 : 1;
  const int mb = (int)((M + 16 * G - 1) / (16 * G));
  note_launch();
  k_lora_prep<RP><<<(int)((N + K + 255) / 256), 256, 0, stream>>>(A, B, r, K, N, 1, 0, at_ws,
                                                                    bt_ws);
  note_launch();
  k_lora_down_fwd<RP, G><<<mb, 256, 0, stream>>>(xc, xsf, gx, gx, M, K, at_ws, scale, 1, t_ws);
  cudaError_t e =
      launch_down_dy<RP, false>(dy, gx, gx, M, N, B, r, scale, 1, u_ws, DyQuant{}, stream);
  if (e != cudaSuccess) return e;
  int64_t ns;
  e = launch_ts<RP, false>(dy, nullptr, nullptr, M, N, t_ws, 1, part, &ns, stream);
  if (e != cudaSuccess) return e;
  note_launch();
  k_lora_ts_reduce<<<std::min<int64_t>((N * r + 255) / 256, num_sms * 8), 256, 0, stream>>>(
      part, (int)ns, N, RP, r, nullptr, 1, dB);
  e = launch_ts<RP, true>(nullptr, xc, xsf, M, K, u_ws, 0, part, &ns, stream);
  if (e != cudaSuccess) return e;
  note_launch();
  k_lora_ts_reduce<<<std::min<int64_t>((K * r + 255) / 256, num_sms * 8), 256, 0, stream>>>(
      part, (int)ns, K, RP, r, gx, 0, dA);
  return cudaGetLastError();
}

cudaError_t launch_lora_adapter_grad(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                     int64_t M, int64_t K, const uint16_t* dy, int64_t N,
                                     const uint16_t* A, const uint16_t* B, int r, int rp,
                                     float scale, float* dA, float* dB, uint16_t* at_ws,
                                     uint16_t* bt_ws, uint16_t* t_ws, uint16_t* u_ws, float* part,
                                     int num_sms, cudaStream_t stream) {
  if (rp == 16)
    return adapter_grad_rp<16>(x_codes, x_sf, gx, M, K, dy, N, A, B, r, scale, dA, dB, at_ws,
                               bt_ws, t_ws, u_ws, part, num_sms, stream);
  if (rp == 32)
    return adapter_grad_rp<32>(x_codes, x_sf, gx, M, K, dy, N, A, B, r, scale, dA, dB, at_ws,
                               bt_ws, t_ws, u_ws, part, num_sms, stream);
  return adapter_grad_rp<64>(x_codes, x_sf, gx, M, K, dy, N, A, B, r, scale, dA, dB, at_ws,
                             bt_ws, t_ws, u_ws, part, num_sms, stream);
}

}  // namespace pact
