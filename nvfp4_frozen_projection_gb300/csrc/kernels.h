// Internal launcher interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "status.h"

namespace pact {

// Counts one kernel launch (pact_launch_count); called before every <<<>>>.
void note_launch();

// Sets the thread's pact_last_error() text and returns code.
int report_error(int code, const char* msg);

struct GemmParams {
  const uint8_t* sfa;      // A scale atoms (128x4 layout, pad4(K/16) blocks per row)
  const uint8_t* sfb;      // B scale atoms
  const float* ga;         // per-tensor scale of A (device)
  const float* gb;         // per-tensor scale of B (device)
  const uint16_t* addend;  // BF16 [M, N] added before the cast, or null (may alias out)
  uint16_t* out;           // BF16 [M, N]
  unsigned* out_amax;      // max |out| as FP32 bits, or null
  unsigned* status;        // device status word
  int M, N, K;             // out [M, N], reduction over K
  int k16p;                // pad4(K/16)
  int num_m, num_n;        // tile grid
  int lora_steps;          // K=16 BF16 MMAs of the LoRA product per tile (0 = none)
  int band_mc;             // tile order: bands of band_mc M-units, each swept over all N
  int addend32;            // addend 32-byte aligned: fetched with 32-byte loads
  int gu_half;             // > 0: the fused gate|up forward in the interleaved column
                           // order; tiles are stored back in the logical order
  unsigned* amax3;         // gu_half > 0 (or null): max |h|, max |gate|, max |up| of the
                           // BF16 output as FP32 bits, h = silu(gate) * up by the exact
                           // FP32 recipe
};

struct GemmLaunch {
  CUtensorMap tmA, tmB, tmLA, tmLB, tmOut;
  CUtensorMap tmSFA, tmSFB;  // scale-factor atoms: rows = 128-row blocks, 8-byte elements
  GemmParams p;
  int num_sms;
};

// Tile width (128 or 256) for an output of N columns and a LoRA operand of rpe
// columns, and the launcher.
int gemm_block_n(int64_t N, int rpe);
// CTAs per cluster along M: 2 when the tile is computed by a CTA pair, else 1.
int gemm_cluster_m(int64_t M, int64_t N, int rpe);
// Bytes of K per A/B tile row in one ring stage (the TMA box width; 64 -> 64B
// swizzle, 128 -> 128B swizzle).
int gemm_stage_row_bytes();
// Whether tiles are computed by CTA pairs (.cta_group::2): each CTA then holds half
// of the B and LoRA up-projection rows of a tile (their tensor-map boxes are bn/2).
bool gemm_uses_pair(int64_t M, int64_t N, int rpe);
cudaError_t launch_gemm_nvfp4(const GemmLaunch& L, int bn, int rpe, int cm, cudaStream_t stream);
cudaError_t status_word_ptr(unsigned** ptr);
// 2-D tiled tensor map over a row-major [rows, inner] matrix of elem_bytes elements
// whose rows are ld elements apart (ld = inner when 0); PACT_OK or an error code (the
// message in pact_last_error).
int make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
             uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
             CUtensorMapSwizzle swz, uint64_t ld = 0);
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_bounds_check(cudaStream_t stream);

// amax pass alone (contiguous rows): max |x| as FP32 bits into *ws_amax.
cudaError_t launch_amax_bf16(const uint16_t* x, int64_t M, int64_t K, unsigned* ws_amax,
                             int num_sms, cudaStream_t stream);
// tmx: BF16 map over x [M, K] (row stride ldx), box 64 x 32, 128-byte swizzle.
cudaError_t launch_quant_bf16(const CUtensorMap& tmx, const uint16_t* x, int64_t M, int64_t K,
                              int64_t ldx, const float* amax_opt, uint8_t* codes, uint8_t* sf,
                              float* g, unsigned* ws_amax, unsigned* status, int num_sms,
                              cudaStream_t stream);
// gu_half > 0: forward layout in the interleaved gate|up row order (gu_interleaved).
cudaError_t launch_pack_weight(const float* W, int64_t N, int64_t K, int backward,
                               int64_t gu_half, uint8_t* codes, uint8_t* sf, float* g,
                               unsigned* ws_amax, int num_sms, cudaStream_t stream);

// LoRA down-projections (BF16 tensor cores, FP32 accumulate), written pre-scaled
// as the left LoRA operand [M, 2 rp] (hi/lo BF16 pair) of the fused GEMM, plus
// the padded right operand [rows, rp].  The forward also needs at_ws [rp, K] of
// workspace for the transposed adapter.
// gu_half > 0: bt_out rows in the interleaved gate|up order (row n = column
// gu_logical(n) of B).
cudaError_t launch_lora_down_fwd(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                 const float* gw, int64_t M, int64_t K, const uint16_t* A,
                                 const uint16_t* B, int r, int rp, float scale, int64_t N,
                                 int64_t gu_half, uint16_t* t_out, uint16_t* bt_out,
                                 uint16_t* at_ws, cudaStream_t stream);
cudaError_t launch_lora_down_dgrad(const uint16_t* dy, const float* gdy, const float* gw,
                                   int64_t M, int64_t N, const uint16_t* A, const uint16_t* B,
                                   int r, int rp, float scale, int64_t K, uint16_t* u_out,
                                   uint16_t* ap_out, cudaStream_t stream);

// (launch_lora_down_dgrad: ap_out null skips the padded copy of A, for r == rp.)
// The same down-projection fused with the NVFP4 quantisation of dY (bit-identical
// to launch_quant_bf16 and launch_lora_down_dgrad): codes/sf/g of dYq and u_out in
// one pass over dY.  amax_opt (device) or ws_amax (filled here by an amax pass).
cudaError_t launch_quant_lora_down(const uint16_t* dy, int64_t M, int64_t N, const float* amax_opt,
                                   unsigned* ws_amax, const float* gw, const uint16_t* A,
                                   const uint16_t* B, int r, int rp, float scale, int64_t K,
                                   uint8_t* codes, uint8_t* sf, float* g, uint16_t* u_out,
                                   uint16_t* ap_out, int num_sms, cudaStream_t stream);
// LoRA adapter gradients dA [K, r] and dB [r, N] (FP32, overwritten).  Workspace:
// at_ws [rp, K] and bt_ws [N, rp] (adapter layouts), t_ws and u_ws [M, 2 rp] BF16,
// part [splits][max(N, K) rp] FP32 with splits = max over the two products of
// lora_ts_splits(M, N, rp, false) and lora_ts_splits(M, K, rp, true).
int64_t lora_ts_splits(int64_t M, int64_t C, int rp, bool fp4, int64_t* rows_per_split);
cudaError_t launch_lora_adapter_grad(const uint8_t* x_codes, const uint8_t* x_sf, const float* gx,
                                     int64_t M, int64_t K, const uint16_t* dy, int64_t N,
                                     const uint16_t* A, const uint16_t* B, int r, int rp,
                                     float scale, float* dA, float* dB, uint16_t* at_ws,
                                     uint16_t* bt_ws, uint16_t* t_ws, uint16_t* u_ws, float* part,
                                     int num_sms, cudaStream_t stream);

// tmx: BF16 map over x [M, H], box 64 x 32, 128-byte swizzle.
cudaError_t launch_rmsnorm_quant(const CUtensorMap& tmx, const uint16_t* x,
                                 const uint16_t* gamma, int64_t M,
                                 int64_t H, float eps, uint8_t* codes, uint8_t* sf, float* g,
                                 float* rstd, unsigned* ws_amax, unsigned* status, int num_sms,
                                 cudaStream_t stream);
cudaError_t launch_silu_mul_quant(const uint16_t* gateup, int64_t M, int64_t I,
                                  const float* amax3_opt, uint8_t* const codes[3],
                                  uint8_t* const sf[3], float* const g[3], unsigned* ws_amax3,
                                  int num_sms, cudaStream_t stream);
cudaError_t launch_silu_mul_bwd(const uint8_t* gc, const uint8_t* gsf, const float* gg,
                                const uint8_t* uc, const uint8_t* usf, const float* ug,
                                const uint16_t* dh, int64_t M, int64_t I, uint16_t* dgu,
                                unsigned* out_amax, int num_sms, cudaStream_t stream);
cudaError_t launch_rmsnorm_bwd(const uint8_t* yc, const uint8_t* ysf, const float* yg,
                               const uint16_t* gamma, const float* rstd, const uint16_t* dy,
                               const uint16_t* dres, int64_t M, int64_t H, uint16_t* dx,
                               unsigned* out_amax, int num_sms, cudaStream_t stream);
cudaError_t launch_pexp(const float* x, float* y, int64_t n, cudaStream_t stream);

}  // namespace pact
