/*
 * libpact — NVFP4 LoRA linear layer for GB300 (sm_103a): C ABI.
 *
 * The method: "PACT: NVFP4 Data-Flow LoRA Fine-Tuning on Consumer GPUs".
 *   Table 6  NVFP4 format: E2M1 elements, one E4M3 scale per block of 16 elements.
 *   Table 7  Precision allocation: frozen projections are NVFP4 GEMMs with FP32
 *            accumulation and BF16 output, backed by cached forward and backward
 *            NVFP4 weight layouts; RMSNorm keeps its NVFP4 output and an FP32
 *            per-token statistic; SiLU-multiply keeps separate NVFP4 gate/up
 *            copies; the LoRA branch runs BF16 GEMMs on the reconstructed shared
 *            input; residual gradients accumulate in BF16.
 *   Figure 3 The LoRA linear layer's forward and backward paths.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory.  Scratch ("ws") is passed in by the caller; its
 *     size comes from the matching *_workspace_size() query and it must be 256-byte
 *     aligned.  The contents of ws need not be initialised.
 *   - All calls are asynchronous on the given CUDA stream (0 = legacy default
 *     stream) and never synchronise the host.  Per-tensor scales stay on the
 *     device.
 *   - BF16 tensors are passed as uint16_t bit patterns, row-major.
 *   - A call validates its arguments on the host and returns a pact_status without
 *     launching anything when they are invalid; pact_last_error() then describes
 *     the problem (thread-local).  A launch failure returns PACT_ERR_CUDA.
 *   - Errors raised inside a kernel (a bounded wait that ran out) are recorded in
 *     a device status word that pact_check_status() reads.
 *   - Outputs must not alias inputs unless a call says so.
 *   - Floating-point inputs are finite.  The debug build (libpact_debug.so) rejects
 *     a NaN: the kernels that quantise, normalise or take an output amax record it
 *     in the status word, and pact_check_status returns PACT_ERR_DEVICE_STATUS.
 *     The release build does not look; a NaN or an infinity there gives
 *     unspecified output values (codes, scales and per-tensor scales included),
 *     but every call still stays within its buffers and ends: no value steers an
 *     address or a loop bound.
 */
#ifndef PACT_H
#define PACT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pact_stream_t; /* a cudaStream_t */

typedef enum pact_status {
  PACT_OK = 0,
  PACT_ERR_INVALID_ARG = 1,  /* null pointer, bad rank, workspace too small, ... */
  PACT_ERR_SHAPE = 2,        /* a dimension breaks the call's divisibility rule */
  PACT_ERR_ALIGN = 3,        /* a pointer breaks the call's alignment rule */
  PACT_ERR_ARCH = 4,         /* the current device is not sm_103 */
  PACT_ERR_CUDA = 5,         /* a CUDA runtime or driver call failed */
  PACT_ERR_TIMEOUT = 6,      /* a kernel's bounded wait ran out (pact_check_status) */
  PACT_ERR_DEVICE_STATUS = 7 /* another kernel-side check failed (pact_check_status) */
} pact_status;

/*
 * An NVFP4 tensor X [rows, cols] (Table 6), cols % 16 == 0:
 *   codes  u8 [rows, cols/2], row stride cols/2 bytes; two E2M1 codes per byte,
 *          the even column in the low nibble.  Code = sign*8 + index of the
 *          magnitude in {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   sf     u8 E4M3 block scales in the layout the block-scaled tensor-core MMA
 *          reads: atoms of 128 rows x 4 blocks (512 bytes) ordered row-block
 *          major, with C16p = pad4(cols/16):
 *            offset(r, c) = ((r/128)*(C16p/4) + c/4)*512 + (r%32)*16
 *                           + ((r%128)/32)*4 + c%4,
 *          pad128(rows) * C16p bytes in total; pad entries are zero.
 *   g      device pointer to the FP32 per-tensor scale.
 * Value of element (r, c):  e2m1(code) * e4m3(sf) * g.
 * codes and sf must be 16-byte aligned (128-byte aligned for GEMM operands).
 */
typedef struct pact_nvfp4 {
  void* codes;
  void* sf;
  float* g;
  int64_t rows;
  int64_t cols;
} pact_nvfp4;

/* Bytes of the code array and of the scale array of an NVFP4 [rows, cols] tensor. */
size_t pact_nvfp4_codes_bytes(int64_t rows, int64_t cols);
size_t pact_nvfp4_sf_bytes(int64_t rows, int64_t cols);

/*
 * Activation quantisation to NVFP4 (Table 6 format; Table 7: both GEMM operands
 * are NVFP4, so X and dY are quantised before the frozen-projection GEMMs).
 *   amax_t = max |x|;  g = amax_t / (6*448);  per block of 16 along a row:
 *   s = e4m3_rne_satfinite(amax_blk / (6*g));  t = e4m3(s)*g;
 *   q = e2m1_rne_satfinite(x / t)  (one IEEE division per element, rounded to
 *   nearest; signed zero codes when t == 0).
 * x: BF16 [M, K], row stride ldx elements (ldx >= K, ldx % 8 == 0), 16-byte aligned.
 * amax_opt: optional device pointer to a precomputed amax_t (skips the first pass).
 * out: codes/sf/g preallocated for [M, K]; out->rows == M, out->cols == K.
 * Rules: M >= 1, K % 64 == 0, pad128(M) * K / 16 < 2^31.
 * ws: pact_quant_nvfp4_workspace_size() bytes.
 */
size_t pact_quant_nvfp4_workspace_size(int64_t M, int64_t K);
int pact_quant_nvfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                     const float* amax_opt, pact_nvfp4* out, void* ws, size_t ws_bytes,
                     pact_stream_t stream);

/*
 * Offline pack of the frozen weight W [N, K] (FP32, row-major; Y = X W^T) into the
 * cached NVFP4 layouts (abstract: "cached forward and backward weight layouts";
 * Table 7 "State retained for backward").  One E4M3 scale per 16x16 tile of W
 * (RTN, g = amax(W)/2688), so both layouts hold the same effective weights:
 *   forward layout  [N, K], blocks of 16 along K  (B operand of Y = X W^T)
 *   backward layout [K, N], blocks of 16 along N  (B operand of dX = dY W)
 * and dequant(backward) == dequant(forward)^T exactly.
 * Rules: N % 64 == 0, K % 64 == 0, W 16-byte aligned.
 * ws: pact_pack_weight_workspace_size() bytes.
 */
size_t pact_pack_weight_workspace_size(int64_t N, int64_t K);
int pact_pack_weight_fwd(const float* W, int64_t N, int64_t K, pact_nvfp4* out_fwd,
                         void* ws, size_t ws_bytes, pact_stream_t stream);
int pact_pack_weight_bwd(const float* W, int64_t N, int64_t K, pact_nvfp4* out_bwd,
                         void* ws, size_t ws_bytes, pact_stream_t stream);

/*
 * Forward pack of a fused gate|up weight W [2I, K] (rows [0, I) gate, [I, 2I) up;
 * Table 7 "SiLU-multiply" and the fused gate/up projection) for
 * pact_lora_linear_fwd_gate_up: the same codes, tile scales and g as
 * pact_pack_weight_fwd, with the rows reordered in groups of 32, a gate group then
 * the matching up group (packed row 64 j + i is gate row 32 j + i, packed row
 * 64 j + 32 + i is up row 32 j + i), so that a GEMM tile holds matching gate and up
 * columns.  The backward layout is unchanged (pact_pack_weight_bwd).
 * Rules as for pact_pack_weight_fwd; N = 2I, N % 64 == 0.
 */
int pact_pack_weight_fwd_gate_up(const float* W, int64_t N, int64_t K, pact_nvfp4* out_fwd,
                                 void* ws, size_t ws_bytes, pact_stream_t stream);

/*
 * LoRA linear forward (Table 7 rows "Frozen projections" and "LoRA branch";
 * Figure 3):
 *   Y = g_x g_w (Xq Wq^T) + scale * (Xhat A) B   [+ residual]
 * with FP32 accumulation and BF16 output; Xhat = dequant(Xq) is the shared NVFP4
 * input of both branches.  The NVFP4 GEMM runs on tcgen05 block-scaled tensor
 * cores; the LoRA product is fused into the same accumulator.
 *   xq     NVFP4 [M, K];  w_fwd NVFP4 [N, K] (forward layout)
 *   A      BF16 [K, r];   B BF16 [r, N];  1 <= r <= 64;  scale = alpha / r
 *   residual_opt  BF16 [M, N] added in FP32 before the BF16 cast (may alias y)
 *   y      BF16 [M, N] output
 *   out_amax_opt  if non-null, receives max |y| over the BF16 output
 * Rules: M >= 1, K % 64 == 0, N % 64 == 0; all pointers 16-byte aligned, NVFP4
 * codes/sf 128-byte aligned.  ws: pact_lora_linear_fwd_workspace_size() bytes.
 */
size_t pact_lora_linear_fwd_workspace_size(int64_t M, int64_t N, int64_t K, int r);
int pact_lora_linear_fwd(const pact_nvfp4* xq, const pact_nvfp4* w_fwd, const uint16_t* A,
                         const uint16_t* B, int r, float scale, const uint16_t* residual_opt,
                         uint16_t* y, float* out_amax_opt, void* ws, size_t ws_bytes,
                         pact_stream_t stream);

/*
 * LoRA linear forward that allocates nothing and needs no workspace.  The paper
 * has no counterpart: this is an interface for callers that cannot allocate
 * device memory or hand in a workspace.  Examples: a plugin whose host framework
 * passes it only inputs and outputs, code running while a stream is captured into
 * a CUDA graph (cudaMalloc is not allowed then), or a runtime with a fixed memory
 * budget where an allocation on the hot path would synchronise the device.
 *
 * Same arguments, rules and result as pact_lora_linear_fwd, without ws/ws_bytes.
 * The scratch lives in a fixed array of PACT_NOALLOC_SCRATCH_BYTES (16 MiB) that
 * is part of the library image; every GPU that loads libpact holds it until the
 * process exits.  A call needs pact_lora_linear_fwd_workspace_size(M, N, K, r) =
 * align256(4 M rp) + align256(2 N rp) + align256(2 K rp) bytes of it (rp = r padded
 * to 16, 32 or 64; align256 rounds up to a multiple of 256); one needing more than
 * 16 MiB returns PACT_ERR_SHAPE without launching anything.
 * - The first call on each device looks up the array's device address (with that
 *   device current) and keeps it for the rest of the process; make that first call
 *   before any stream capture.  The kept address assumes the device's context lives
 *   as long as the process: after cudaDeviceReset() on a device, do not call this
 *   entry point on that device again.
 * - Every call shares the one array, so calls that overlap on the GPU (different
 *   streams, or different host threads) race and corrupt each other's results.
 *   Serialise them, e.g. issue them all on one stream.
 */
#define PACT_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
size_t pact_lora_linear_fwd_noalloc_max_scratch(void);
int pact_lora_linear_fwd_noalloc(const pact_nvfp4* xq, const pact_nvfp4* w_fwd,
                                 const uint16_t* A, const uint16_t* B, int r, float scale,
                                 const uint16_t* residual_opt, uint16_t* y, float* out_amax_opt,
                                 pact_stream_t stream);

/*
 * LoRA linear input gradient (Table 7: "NVFP4 input-gradient GEMMs" on the cached
 * backward layout; LoRA branch "BF16 ... input gradients"):
 *   dX = g_dy g_w (dYq Wbwd^T) + scale * (dY B^T) A^T   [+ dX_prev if accumulate]
 *   dyq    NVFP4 [M, N];  dy BF16 [M, N] (the same gradient before quantisation,
 *          used by the BF16 LoRA branch);  w_bwd NVFP4 [K, N] (backward layout)
 *   A BF16 [K, r];  B BF16 [r, N];  1 <= r <= 64;  scale = alpha / r
 *   accumulate  0: dx = result;  1: dx += result (BF16 gradient accumulation,
 *               e.g. the q/k/v input gradients summed into one dX)
 *   dx     BF16 [M, K] output
 * Rules as for the forward.  ws: pact_lora_linear_dgrad_workspace_size() bytes.
 */
/*
 * The fused gate|up projection's forward with the statistics of its output that the
 * SiLU-multiply quantisation needs (Table 7 "SiLU-multiply": NVFP4 h and separate
 * NVFP4 gate/up copies, each with its own per-tensor scale), produced by the GEMM
 * epilogue so that pact_silu_mul_quant runs as one pass:
 *   y = [gate | up] as pact_lora_linear_fwd computes it, bit for bit, in the logical
 *       column order (gate columns [0, I), up columns [I, 2I));
 *   amax3[0] = max |h|, h = silu(gate) * up by the SiLU-multiply's exact FP32
 *   recipe on the BF16 values of y; amax3[1] = max |gate|, amax3[2] = max |up|;
 *   the layout pact_silu_mul_quant takes as amax3_opt.
 *   w_fwd_gu: pact_pack_weight_fwd_gate_up's layout;  A [K, r], B [r, 2I]: the fused
 *   adapters in the logical order (B block-diagonal for separate gate and up
 *   adapters);  amax3: device FP32 [3], 4-byte aligned, overwritten.
 * Rules and workspace as for pact_lora_linear_fwd (no residual); N = 2I, N % 64 == 0.
 */
int pact_lora_linear_fwd_gate_up(const pact_nvfp4* xq, const pact_nvfp4* w_fwd_gu,
                                 const uint16_t* A, const uint16_t* B, int r, float scale,
                                 uint16_t* y, float* amax3, void* ws, size_t ws_bytes,
                                 pact_stream_t stream);

size_t pact_lora_linear_dgrad_workspace_size(int64_t M, int64_t N, int64_t K, int r);
int pact_lora_linear_dgrad(const pact_nvfp4* dyq, const uint16_t* dy, const pact_nvfp4* w_bwd,
                           const uint16_t* A, const uint16_t* B, int r, float scale,
                           int accumulate, uint16_t* dx, void* ws, size_t ws_bytes,
                           pact_stream_t stream);

/*
 * LoRA linear input gradient with the quantisation of dY fused in: the same result
 * as pact_quant_nvfp4(dy, M, N, N, dy_amax_opt, dyq_out, ...) followed by
 * pact_lora_linear_dgrad(dyq_out, dy, w_bwd, ...) (the same bytes in dyq_out, the
 * same dx), with one pass over dY fewer: one kernel encodes dY to NVFP4 and forms
 * the LoRA down-projection dY B^T from the same loads.
 *   dy BF16 [M, N], contiguous rows;  dy_amax_opt: optional device FP32 max |dy|
 *   (e.g. a producer's out_amax; without it an amax pass runs first);
 *   dyq_out NVFP4 [M, N], caller-owned, written (codes, every scale byte of the
 *   padded atoms, g) and left for reuse;  the other arguments as for
 *   pact_lora_linear_dgrad.
 * Rules as for pact_lora_linear_dgrad, plus pad128(M) * N / 64 < 2^31.
 * ws: pact_lora_linear_dgrad_q_workspace_size() bytes, 256-byte aligned.
 */
size_t pact_lora_linear_dgrad_q_workspace_size(int64_t M, int64_t N, int64_t K, int r);
int pact_lora_linear_dgrad_q(const uint16_t* dy, const float* dy_amax_opt,
                             const pact_nvfp4* w_bwd, const uint16_t* A, const uint16_t* B, int r,
                             float scale, int accumulate, pact_nvfp4* dyq_out, uint16_t* dx,
                             void* ws, size_t ws_bytes, pact_stream_t stream);

/*
 * LoRA adapter gradients (Table 7: LoRA branch "BF16 adapter gradients"; Figure 1,
 * the trainable A, B beside the frozen NVFP4 projection).  With Xhat the dequantised
 * NVFP4 input that the forward multiplied (the tensor retained for backward):
 *   dA = scale * Xhat^T (dY B^T)      FP32 [K, r]
 *   dB = scale * (Xhat A)^T dY        FP32 [r, N]
 *   xq  NVFP4 [M, K] (the forward's xq);  dy BF16 [M, N] (the output gradient before
 *       quantisation, as passed to pact_lora_linear_dgrad);  A BF16 [K, r];
 *   B BF16 [r, N];  1 <= r <= 64;  scale = alpha / r;  N the output width.
 *   dA, dB are overwritten (not accumulated).
 * Arithmetic: dY B^T and Xhat A are formed in FP32 and carried as a hi + lo pair of
 * BF16 values (about 16 significant bits); the products with Xhat (exact in BF16
 * once the per-tensor scale is factored out) and dY accumulate in FP32 over row
 * splits whose partial sums are added in a fixed order, so results are
 * deterministic run to run.
 * Rules: M >= 1, N and K multiples of 64; dy and B 16-byte, dA and dB 4-byte
 * aligned; xq codes/sf 16-byte aligned.  ws: pact_lora_adapter_grad_workspace_size()
 * bytes, 256-byte aligned, owned by the caller and free again when the stream
 * reaches the end of the call.  Errors are reported before any launch.
 */
size_t pact_lora_adapter_grad_workspace_size(int64_t M, int64_t N, int64_t K, int r);
int pact_lora_adapter_grad(const pact_nvfp4* xq, const uint16_t* dy, const uint16_t* A,
                           const uint16_t* B, int r, float scale, int64_t N, float* dA,
                           float* dB, void* ws, size_t ws_bytes, pact_stream_t stream);

/*
 * Fused RMSNorm -> NVFP4 (abstract: "reuses quantized RMSNorm outputs"; Table 7
 * "RMSNorm": BF16 input, FP32 normalisation, retains the NVFP4 output and the FP32
 * per-token statistic).  Per row:
 *   ss by a fixed order (row split in blocks of 16; lane l = 0..31 sums blocks
 *   l, l+32, ... element by element; butterfly over offsets 16, 8, 4, 2, 1);
 *   rstd = 1 / sqrt(ss/H + eps);  y_j = (x_j * rstd) * gamma_j   (FP32);
 * then y (FP32, never rounded to BF16) is quantised like pact_quant_nvfp4.
 *   x BF16 [M, H];  gamma BF16 [H];  yq NVFP4 [M, H] out;  rstd FP32 [M] out.
 * Rules: M >= 1, H % 64 == 0, H <= 16384, pad128(M) * H / 16 < 2^31.
 * ws: pact_rmsnorm_quant_workspace_size().
 */
size_t pact_rmsnorm_quant_workspace_size(int64_t M, int64_t H);
int pact_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t H,
                       float eps, pact_nvfp4* yq, float* rstd, void* ws, size_t ws_bytes,
                       pact_stream_t stream);

/*
 * Fused SiLU-multiply -> NVFP4 (abstract: "saves gate/up activations in NVFP4";
 * Table 7 "SiLU-multiply": BF16 gate/up inputs, FP32 arithmetic, separate NVFP4
 * gate/up copies retained for backward).
 *   gateup BF16 [M, 2I]: gate = columns [0, I), up = columns [I, 2I).
 *   h = (gate / (1 + exp(-gate))) * up in FP32, with exp evaluated by the fixed
 *   recipe of pact_test_pexp; hq = NVFP4(h); gate_q = NVFP4(gate); up_q = NVFP4(up),
 *   each with its own per-tensor scale.
 *   amax3_opt: optional device FP32[3] = {amax(h), amax(gate), amax(up)}.
 * Rules: M >= 1, I % 64 == 0.  ws: pact_silu_mul_quant_workspace_size() bytes.
 */
size_t pact_silu_mul_quant_workspace_size(int64_t M, int64_t I);
int pact_silu_mul_quant(const uint16_t* gateup, int64_t M, int64_t I, const float* amax3_opt,
                        pact_nvfp4* hq, pact_nvfp4* gate_q, pact_nvfp4* up_q, void* ws,
                        size_t ws_bytes, pact_stream_t stream);

/*
 * SiLU-multiply backward (Table 7: FP32 reconstruction from the NVFP4 gate/up
 * copies and derivatives, BF16 gradients).  With g, u the dequantised copies and
 * s = 1/(1+exp(-g)):  dgate = dh*u*s*(1 + g*(1-s)),  dup = dh*g*s.
 *   gate_q, up_q NVFP4 [M, I];  dh BF16 [M, I];  dgateup BF16 [M, 2I] out
 *   (dgate in columns [0, I), dup in [I, 2I)).
 *   out_amax_opt: if non-null receives max |dgateup| (BF16 values), for a
 *   following single-pass pact_quant_nvfp4.
 * Rules: M >= 1, I % 64 == 0.
 */
int pact_silu_mul_bwd(const pact_nvfp4* gate_q, const pact_nvfp4* up_q, const uint16_t* dh,
                      uint16_t* dgateup, float* out_amax_opt, pact_stream_t stream);

/*
 * RMSNorm backward (Table 7: FP32 reconstruction and reduction, BF16 gradient):
 * n = dequant(yq)/gamma, dn = dy*gamma, c = sum_j(dn_j n_j)/H,
 * dx = rstd*(dn - n*c)  [+ dres]  (dres: residual-stream gradient, BF16 addition).
 *   yq NVFP4 [M, H] (the forward output);  gamma BF16 [H];  rstd FP32 [M];
 *   dy BF16 [M, H];  dres_opt BF16 [M, H] or NULL (may alias dx);  dx BF16 [M, H].
 *   out_amax_opt: if non-null (4-byte aligned, device) receives max |dx| over the
 *   BF16 outputs, so that a following pact_quant_nvfp4 of dx is single-pass.
 * Rules: M >= 1, H % 64 == 0, H <= 16384.
 */
int pact_rmsnorm_bwd(const pact_nvfp4* yq, const uint16_t* gamma, const float* rstd,
                     const uint16_t* dy, const uint16_t* dres_opt, uint16_t* dx,
                     float* out_amax_opt, pact_stream_t stream);

/*
 * The FP32 exp recipe used by pact_silu_mul_quant, exposed so that it can be
 * compared bit for bit with another implementation: Cody-Waite reduction
 * x = n ln2 + f (ln2 split in a 16-bit head and a tail), degree-7 Taylor
 * polynomial of e^f by Horner's rule with fused multiply-adds, exact scaling by
 * 2^n; +inf above 0x1.62e42ep+6, 0 below -0x1.9fe368p+6.  x, y FP32 [n] (device).
 */
int pact_test_pexp(const float* x, float* y, int64_t n, pact_stream_t stream);

/*
 * Measurement hooks (no counterpart in the method; host-side bookkeeping only).
 * pact_launch_count: number of libpact kernels launched by this process so far
 *   (launches replayed from a captured CUDA graph are not counted again).
 * pact_profile_next_gemm: arm a one-shot recording of two caller-created CUDA
 *   events (cudaEvent_t, passed as void*) on the launch stream immediately before
 *   and after the next NVFP4 GEMM kernel launched by this host thread, so that
 *   the kernel can be timed without the LoRA down-projection launched beside it.
 *   Pass NULLs to disarm.
 */
uint64_t pact_launch_count(void);
int pact_profile_next_gemm(void* begin_event, void* end_event);

/*
 * Test of the failure path (no counterpart in the method).  Launches one thread
 * that waits, with the bounded wait the GEMM kernels use, on a barrier that nothing
 * completes; after limit_us microseconds (1 .. 2e6) it records a timeout in the
 * device status word and returns.  pact_check_status() then reports
 * PACT_ERR_TIMEOUT, and the context stays usable.
 */
int pact_test_wait_timeout(uint32_t limit_us, pact_stream_t stream);

/*
 * Test of the debug build's bounds checks (no counterpart in the method).  The
 * library built with -DPACT_DEBUG (libpact_debug.so) checks the index of every
 * store whose address it computes by hand against the buffer's extent; a failed
 * check skips the store and records PACT_DEV_BOUNDS in the device status word
 * instead of trapping.  This launches one thread that evaluates one failing check
 * and accesses no memory: afterwards pact_check_status() reports
 * PACT_ERR_DEVICE_STATUS in the debug build and PACT_OK in the release build, whose
 * checks compile away.
 */
int pact_test_bounds_check(pact_stream_t stream);

/* Synchronises the stream, then returns and clears the device status word:
 * PACT_OK, PACT_ERR_TIMEOUT or PACT_ERR_DEVICE_STATUS.  For tests and debugging. */
int pact_check_status(pact_stream_t stream);

/* PACT_OK when the current CUDA device is sm_103 (GB300), else PACT_ERR_ARCH. */
int pact_device_supported(void);

/* Description of the last error returned on this host thread ("" if none). */
const char* pact_last_error(void);

/* Library version string. */
const char* pact_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PACT_H */
