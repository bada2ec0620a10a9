// C ABI of libpact: argument validation, workspace carving, TMA descriptors and
// kernel launches.  Declarations and the contract of every call are in pact.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/pact.h"
#include "kernels.h"

using namespace pact;

namespace {
std::atomic<uint64_t> g_launches{0};
thread_local cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;
}  // namespace

void pact::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
int fail(int code, const char* fmt, ...);
}

int pact::report_error(int code, const char* msg) { return fail(code, "%s", msg); }

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PACT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int major = 0, minor = 0;
  unsigned* status = nullptr;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(PACT_ERR_INVALID_ARG, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "multiprocessor count");
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if ((e = status_word_ptr(&d.status)) != cudaSuccess) return cuda_fail(e, "status word");
    d.init = true;
  }
  if (!(d.major == 10 && d.minor == 3))
    return fail(PACT_ERR_ARCH, "device is sm_%d%d; libpact needs sm_103 (GB300)", d.major,
                d.minor);
  *out = &d;
  return PACT_OK;
}

// ---------------------------------------------------------------- TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// 2-D tiled map over a row-major [rows, inner] matrix of elem-byte elements whose
// rows are ld elements apart (ld = inner when 0).
int pact::make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
             uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
             CUtensorMapSwizzle swz, uint64_t ld) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(PACT_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {(ld ? ld : inner) * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PACT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PACT_OK;
}

namespace {

// ---------------------------------------------------------------- validation helpers
int64_t pad_to(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int check_nvfp4(const pact_nvfp4* t, const char* name, int64_t rows, int64_t cols, uintptr_t al) {
  if (!t) return fail(PACT_ERR_INVALID_ARG, "%s is null", name);
  if (!t->codes || !t->sf || !t->g) return fail(PACT_ERR_INVALID_ARG, "%s has a null field", name);
  if (t->rows != rows || t->cols != cols)
    return fail(PACT_ERR_SHAPE, "%s is [%lld, %lld], expected [%lld, %lld]", name,
                (long long)t->rows, (long long)t->cols, (long long)rows, (long long)cols);
  if (!aligned(t->codes, al) || !aligned(t->sf, al) || !aligned(t->g, 4))
    return fail(PACT_ERR_ALIGN, "%s codes/sf must be %d-byte aligned", name, (int)al);
  return PACT_OK;
}

// LoRA rank padded to 16, 32 or 64; the fused GEMM's LoRA operands are twice as
// wide (a hi/lo BF16 pair of the down-projection output).
int rp_for(int r) { return r <= 16 ? 16 : (r <= 32 ? 32 : 64); }

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* pact_last_error(void) { return g_err; }

#ifdef PACT_DEBUG
const char* pact_version(void) { return "libpact 0.2 (sm_103a, debug: bounds-checked stores, NaN checks)"; }
#else
const char* pact_version(void) { return "libpact 0.2 (sm_103a)"; }
#endif

uint64_t pact_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pact_profile_next_gemm(void* begin_event, void* end_event) {
  g_prof_begin = (cudaEvent_t)begin_event;
  g_prof_end = (cudaEvent_t)end_event;
  return PACT_OK;
}

int pact_device_supported(void) {
  DeviceInfo* d;
  return device_info(&d);
}

size_t pact_nvfp4_codes_bytes(int64_t rows, int64_t cols) {
  return rows > 0 && cols > 0 ? (size_t)(rows * (cols / 2)) : 0;
}

size_t pact_nvfp4_sf_bytes(int64_t rows, int64_t cols) {
  return rows > 0 && cols > 0 ? (size_t)(pad_to(rows, 128) * pad_to(cols / 16, 4)) : 0;
}

int pact_check_status(pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned v = 0;
  if ((e = cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status word");
  if (v) {
    unsigned zero = 0;
    cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (v & PACT_DEV_TIMEOUT)
      return fail(PACT_ERR_TIMEOUT, "a kernel wait timed out (status 0x%x)", v);
    if (v & PACT_DEV_BOUNDS)
      return fail(PACT_ERR_DEVICE_STATUS, "a bounds check of the debug build failed (status 0x%x)",
                  v);
    if (v & PACT_DEV_NAN)
      return fail(PACT_ERR_DEVICE_STATUS,
                  "the debug build found a NaN among the input values (status 0x%x)", v);
    return fail(PACT_ERR_DEVICE_STATUS, "device status 0x%x", v);
  }
  return PACT_OK;
}

// ---------------------------------------------------------------- quantisation
size_t pact_quant_nvfp4_workspace_size(int64_t, int64_t) { return 256; }

int pact_quant_nvfp4(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* amax_opt,
                     pact_nvfp4* out, void* ws, size_t ws_bytes, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!x) return fail(PACT_ERR_INVALID_ARG, "x is null");
  if (M < 1 || K < 64 || K % 64) return fail(PACT_ERR_SHAPE, "need M >= 1 and K %% 64 == 0");
  if (pad_to(M, 128) * (K / 16) >= (int64_t)1 << 31)
    return fail(PACT_ERR_SHAPE, "tensor too large: pad128(M) * K / 16 must be < 2^31");
  if (ldx < K || ldx % 8) return fail(PACT_ERR_SHAPE, "need ldx >= K and ldx %% 8 == 0");
  if (!aligned(x, 16)) return fail(PACT_ERR_ALIGN, "x must be 16-byte aligned");
  if ((rc = check_nvfp4(out, "out", M, K, 16))) return rc;
  if (!ws || ws_bytes < pact_quant_nvfp4_workspace_size(M, K) || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  CUtensorMap tmx;
  if ((rc = make_map(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, K, M, 64, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B, ldx)))
    return rc;
  cudaError_t e = launch_quant_bf16(tmx, x, M, K, ldx, amax_opt, (uint8_t*)out->codes,
                                    (uint8_t*)out->sf, out->g, (unsigned*)ws, d->status, d->sms,
                                    (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "quant launch");
}

// ---------------------------------------------------------------- weight pack
size_t pact_pack_weight_workspace_size(int64_t, int64_t) { return 256; }

static int pack_common(const float* W, int64_t N, int64_t K, pact_nvfp4* out, void* ws,
                       size_t ws_bytes, pact_stream_t stream, int backward, int64_t gu_half) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!W) return fail(PACT_ERR_INVALID_ARG, "W is null");
  if (N < 64 || K < 64 || N % 64 || K % 64)
    return fail(PACT_ERR_SHAPE, "need N %% 64 == 0 and K %% 64 == 0");
  if (!aligned(W, 16)) return fail(PACT_ERR_ALIGN, "W must be 16-byte aligned");
  if ((rc = check_nvfp4(out, backward ? "out_bwd" : "out_fwd", backward ? K : N, backward ? N : K,
                        16)))
    return rc;
  if (!ws || ws_bytes < 256 || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  cudaError_t e = launch_pack_weight(W, N, K, backward, gu_half, (uint8_t*)out->codes,
                                     (uint8_t*)out->sf, out->g, (unsigned*)ws, d->sms,
                                     (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "pack launch");
}

int pact_pack_weight_fwd(const float* W, int64_t N, int64_t K, pact_nvfp4* out_fwd, void* ws,
                         size_t ws_bytes, pact_stream_t stream) {
  return pack_common(W, N, K, out_fwd, ws, ws_bytes, stream, 0, 0);
}

int pact_pack_weight_fwd_gate_up(const float* W, int64_t N, int64_t K, pact_nvfp4* out_fwd,
                                 void* ws, size_t ws_bytes, pact_stream_t stream) {
  if (N % 64) return fail(PACT_ERR_SHAPE, "need N %% 64 == 0 (gate and up each a multiple of 32)");
  return pack_common(W, N, K, out_fwd, ws, ws_bytes, stream, 0, N / 2);
}

int pact_pack_weight_bwd(const float* W, int64_t N, int64_t K, pact_nvfp4* out_bwd, void* ws,
                         size_t ws_bytes, pact_stream_t stream) {
  return pack_common(W, N, K, out_bwd, ws, ws_bytes, stream, 1, 0);
}

// ---------------------------------------------------------------- LoRA linear
// Workspace: the LoRA left operand [M, 2 rp] (hi|lo BF16 pair) and the padded right
// operand [rows, rp], both BF16; the forward also keeps A^T [rp, K] for its
// down-projection.
size_t pact_lora_linear_fwd_workspace_size(int64_t M, int64_t N, int64_t K, int r) {
  if (M < 1 || N < 1 || K < 1 || r < 1 || r > 64) return 0;
  const int rp = rp_for(r);
  return align256((size_t)M * 2 * rp * 2) + align256((size_t)N * rp * 2) +
         align256((size_t)K * rp * 2);
}

size_t pact_lora_linear_dgrad_workspace_size(int64_t M, int64_t, int64_t K, int r) {
  if (M < 1 || K < 1 || r < 1 || r > 64) return 0;
  const int rp = rp_for(r);
  return align256((size_t)M * 2 * rp * 2) + align256((size_t)K * rp * 2);
}

// Shared tail of fwd and dgrad: GEMM OUT[M, Nout] over reduction Kr with the
// NVFP4 operands a [M, Kr], b [Nout, Kr] and the LoRA operands la [M, rpe],
// lb [Nout, rpe] (both BF16, in the workspace).
static int run_gemm(DeviceInfo* d, const pact_nvfp4* a, const pact_nvfp4* b, int64_t M,
                    int64_t Nout, int64_t Kr, const uint16_t* la, const uint16_t* lb, int rpe,
                    const uint16_t* addend, uint16_t* out, float* out_amax, cudaStream_t stream,
                    int64_t gu_half = 0, float* amax3 = nullptr) {
  GemmLaunch L;
  std::memset(&L, 0, sizeof(L));
  const int bn = gemm_block_n(Nout, rpe);
  const int cm = gemm_cluster_m(M, Nout, rpe);  // each CTA of a cluster loads bn / cm rows of B
  int rc;
  const uint32_t rowb = (uint32_t)gemm_stage_row_bytes();
  const CUtensorMapSwizzle absw = rowb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if ((rc = make_map(&L.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a->codes, Kr / 2, M, rowb, 128,
                     absw)))
    return rc;
  if ((rc = make_map(&L.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b->codes, Kr / 2, Nout, rowb,
                     bn / cm, absw)))
    return rc;
  // LoRA operands: la [M, rpe] (hi|lo pair), lb [Nout, rpe/2]; boxes of at most 64
  // columns (128-byte rows), swizzled by their row width.
  auto lsw = [](uint32_t cols) {
    return cols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                      : (cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
  };
  const uint32_t rp = (uint32_t)rpe / 2;
  const uint32_t abox = rpe < 64 ? (uint32_t)rpe : 64, bbox = rp < 64 ? rp : 64;
  if ((rc = make_map(&L.tmLA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, la, rpe, M, abox, 128,
                     lsw(abox))))
    return rc;
  const uint32_t lb_rows = gemm_uses_pair(M, Nout, rpe) ? (uint32_t)bn / 2 : (uint32_t)bn;
  if ((rc = make_map(&L.tmLB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lb, rp, Nout, bbox, lb_rows,
                     lsw(bbox))))
    return rc;
  // scale factors: each 128-row block is one row of k16p / 4 atoms (512 bytes each),
  // read as 8-byte elements; a stage takes 4 atoms (2 KB) of one A block and of the
  // bn / 128 B blocks of its tile (zero fill past K and past the last block)
  const uint64_t sf_row = (uint64_t)pad_to(Kr / 16, 4) * 16;  // 8-byte elements per block row
  if ((rc = make_map(&L.tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT64, 8, a->sf, sf_row,
                     (uint64_t)pad_to(M, 128) / 128, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE)))
    return rc;
  if ((rc = make_map(&L.tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT64, 8, b->sf, sf_row,
                     (uint64_t)pad_to(Nout, 128) / 128, 256, (uint32_t)bn / 128,
                     CU_TENSOR_MAP_SWIZZLE_NONE)))
    return rc;
  // output: 32 x 32 BF16 blocks written by TMA stores from the epilogue's 64-byte
  // swizzled staging buffers
  if ((rc = make_map(&L.tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, Nout, M, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_64B)))
    return rc;
  GemmParams& p = L.p;
  p.sfa = (const uint8_t*)a->sf;
  p.sfb = (const uint8_t*)b->sf;
  p.ga = a->g;
  p.gb = b->g;
  p.addend = addend;
  p.addend32 = addend && aligned(addend, 32);
  p.out = out;
  p.out_amax = (unsigned*)out_amax;
  p.status = d->status;
  p.M = (int)M;
  p.N = (int)Nout;
  p.K = (int)Kr;
  p.k16p = (int)pad_to(Kr / 16, 4);
  p.num_m = (int)((M + 127) / 128);
  p.num_n = (int)((Nout + bn - 1) / bn);
  p.lora_steps = rpe / 16;
  p.gu_half = (int)gu_half;
  p.amax3 = (unsigned*)amax3;
  L.num_sms = d->sms;
  if (out_amax) {
    cudaError_t e = cudaMemsetAsync(out_amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e, "amax reset");
  }
  if (amax3) {
    cudaError_t e = cudaMemsetAsync(amax3, 0, 3 * sizeof(float), stream);
    if (e != cudaSuccess) return cuda_fail(e, "amax reset");
  }
  cudaEvent_t pb = g_prof_begin, pe = g_prof_end;
  g_prof_begin = g_prof_end = nullptr;
  if (pb && cudaEventRecord(pb, stream) != cudaSuccess) return cuda_fail(cudaGetLastError(), "event");
  cudaError_t e = launch_gemm_nvfp4(L, bn, rpe, cm, stream);
  if (e == cudaSuccess && pe && cudaEventRecord(pe, stream) != cudaSuccess)
    return cuda_fail(cudaGetLastError(), "event");
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "gemm launch");
}

static int check_gemm_dims(int64_t M, int64_t N, int64_t K, int r) {
  if (M < 1 || M > (1 << 30)) return fail(PACT_ERR_SHAPE, "need 1 <= M <= 2^30");
  if (N < 64 || N % 64 || K < 64 || K % 64 || N > (1 << 30) || K > (1 << 30))
    return fail(PACT_ERR_SHAPE, "need N %% 64 == 0 and K %% 64 == 0");
  if (r < 1 || r > 64) return fail(PACT_ERR_INVALID_ARG, "need 1 <= r <= 64");
  return PACT_OK;
}

static int lora_fwd_impl(const pact_nvfp4* xq, const pact_nvfp4* w_fwd, const uint16_t* A,
                         const uint16_t* B, int r, float scale, const uint16_t* residual_opt,
                         uint16_t* y, float* out_amax_opt, void* ws, size_t ws_bytes,
                         pact_stream_t stream, int gate_up, float* amax3) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!xq || !w_fwd) return fail(PACT_ERR_INVALID_ARG, "xq and w_fwd are required");
  const int64_t M = xq->rows, K = xq->cols, N = w_fwd->rows;
  if ((rc = check_gemm_dims(M, N, K, r))) return rc;
  if ((rc = check_nvfp4(xq, "xq", M, K, 128)) || (rc = check_nvfp4(w_fwd, "w_fwd", N, K, 128)))
    return rc;
  if (!A || !B || !y) return fail(PACT_ERR_INVALID_ARG, "A, B and y are required");
  if (!aligned(y, 16) || (residual_opt && !aligned(residual_opt, 16)) || !aligned(B, 2) ||
      !aligned(A, 2))
    return fail(PACT_ERR_ALIGN, "y and residual must be 16-byte aligned");
  if (!ws || ws_bytes < pact_lora_linear_fwd_workspace_size(M, N, K, r) || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  const int rp = rp_for(r);
  const int64_t gu_half = gate_up ? N / 2 : 0;
  if (gate_up && (N % 64 || !amax3 || !aligned(amax3, 4)))
    return fail(PACT_ERR_INVALID_ARG, "gate|up forward: need N %% 64 == 0 and a 4-byte aligned amax3");
  uint16_t* t = (uint16_t*)ws;
  uint16_t* bt = (uint16_t*)((char*)ws + align256((size_t)M * 2 * rp * 2));
  uint16_t* at = (uint16_t*)((char*)bt + align256((size_t)N * rp * 2));
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_lora_down_fwd((const uint8_t*)xq->codes, (const uint8_t*)xq->sf, xq->g,
                                       w_fwd->g, M, K, A, B, r, rp, scale, N, gu_half, t, bt, at,
                                       s);
  if (e != cudaSuccess) return cuda_fail(e, "lora down launch");
  return run_gemm(d, xq, w_fwd, M, N, K, t, bt, 2 * rp, residual_opt, y, out_amax_opt, s, gu_half,
                  amax3);
}

int pact_lora_linear_fwd(const pact_nvfp4* xq, const pact_nvfp4* w_fwd, const uint16_t* A,
                         const uint16_t* B, int r, float scale, const uint16_t* residual_opt,
                         uint16_t* y, float* out_amax_opt, void* ws, size_t ws_bytes,
                         pact_stream_t stream) {
  return lora_fwd_impl(xq, w_fwd, A, B, r, scale, residual_opt, y, out_amax_opt, ws, ws_bytes,
                       stream, 0, nullptr);
}

int pact_lora_linear_fwd_gate_up(const pact_nvfp4* xq, const pact_nvfp4* w_fwd_gu,
                                 const uint16_t* A, const uint16_t* B, int r, float scale,
                                 uint16_t* y, float* amax3, void* ws, size_t ws_bytes,
                                 pact_stream_t stream) {
  return lora_fwd_impl(xq, w_fwd_gu, A, B, r, scale, nullptr, y, nullptr, ws, ws_bytes, stream, 1,
                       amax3);
}

int pact_lora_linear_dgrad(const pact_nvfp4* dyq, const uint16_t* dy, const pact_nvfp4* w_bwd,
                           const uint16_t* A, const uint16_t* B, int r, float scale,
                           int accumulate, uint16_t* dx, void* ws, size_t ws_bytes,
                           pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!dyq || !w_bwd) return fail(PACT_ERR_INVALID_ARG, "dyq and w_bwd are required");
  const int64_t M = dyq->rows, N = dyq->cols, K = w_bwd->rows;
  if ((rc = check_gemm_dims(M, N, K, r))) return rc;
  if ((rc = check_nvfp4(dyq, "dyq", M, N, 128)) || (rc = check_nvfp4(w_bwd, "w_bwd", K, N, 128)))
    return rc;
  if (!dy || !A || !B || !dx) return fail(PACT_ERR_INVALID_ARG, "dy, A, B and dx are required");
  if (!aligned(dx, 16) || !aligned(dy, 16) || !aligned(B, 16) || !aligned(A, 2))
    return fail(PACT_ERR_ALIGN, "dx, dy and B must be 16-byte aligned");
  if (!ws || ws_bytes < pact_lora_linear_dgrad_workspace_size(M, N, K, r) || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  const int rp = rp_for(r);
  uint16_t* u = (uint16_t*)ws;
  uint16_t* ap = (uint16_t*)((char*)ws + align256((size_t)M * 2 * rp * 2));
  // A [K, r] with r == rp is already the zero-padded [K, rp] operand the GEMM reads
  const bool a_direct = r == rp && aligned(A, 16);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_lora_down_dgrad(dy, dyq->g, w_bwd->g, M, N, A, B, r, rp, scale, K, u,
                                         a_direct ? nullptr : ap, s);
  if (e != cudaSuccess) return cuda_fail(e, "lora down launch");
  return run_gemm(d, dyq, w_bwd, M, K, N, u, a_direct ? A : ap, 2 * rp, accumulate ? dx : nullptr,
                  dx, nullptr, s);
}

// ---------------------------------------------------------------- dgrad with dY quantisation
size_t pact_lora_linear_dgrad_q_workspace_size(int64_t M, int64_t N, int64_t K, int r) {
  const size_t w = pact_lora_linear_dgrad_workspace_size(M, N, K, r);
  return w ? w + 256 : 0;
}

int pact_lora_linear_dgrad_q(const uint16_t* dy, const float* dy_amax_opt,
                             const pact_nvfp4* w_bwd, const uint16_t* A, const uint16_t* B, int r,
                             float scale, int accumulate, pact_nvfp4* dyq_out, uint16_t* dx,
                             void* ws, size_t ws_bytes, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!dyq_out || !w_bwd) return fail(PACT_ERR_INVALID_ARG, "dyq_out and w_bwd are required");
  const int64_t M = dyq_out->rows, N = dyq_out->cols, K = w_bwd->rows;
  if ((rc = check_gemm_dims(M, N, K, r))) return rc;
  if (pad_to(M, 128) * (N / 64) >= (int64_t)1 << 31)
    return fail(PACT_ERR_SHAPE, "tensor too large: pad128(M) * N / 64 must be < 2^31");
  if ((rc = check_nvfp4(dyq_out, "dyq_out", M, N, 128)) ||
      (rc = check_nvfp4(w_bwd, "w_bwd", K, N, 128)))
    return rc;
  if (!dy || !A || !B || !dx) return fail(PACT_ERR_INVALID_ARG, "dy, A, B and dx are required");
  if (!aligned(dx, 16) || !aligned(dy, 16) || !aligned(B, 16) || !aligned(A, 2) ||
      (dy_amax_opt && !aligned(dy_amax_opt, 4)))
    return fail(PACT_ERR_ALIGN, "dx, dy and B must be 16-byte aligned");
  if (!ws || ws_bytes < pact_lora_linear_dgrad_q_workspace_size(M, N, K, r) || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  const int rp = rp_for(r);
  uint16_t* u = (uint16_t*)ws;
  uint16_t* ap = (uint16_t*)((char*)ws + align256((size_t)M * 2 * rp * 2));
  unsigned* amax_ws = (unsigned*)((char*)ws + pact_lora_linear_dgrad_workspace_size(M, N, K, r));
  const bool a_direct = r == rp && aligned(A, 16);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_quant_lora_down(dy, M, N, dy_amax_opt, amax_ws, w_bwd->g, A, B, r, rp,
                                         scale, K, (uint8_t*)dyq_out->codes,
                                         (uint8_t*)dyq_out->sf, dyq_out->g, u,
                                         a_direct ? nullptr : ap, d->sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "quant + lora down launch");
  return run_gemm(d, dyq_out, w_bwd, M, K, N, u, a_direct ? A : ap, 2 * rp,
                  accumulate ? dx : nullptr, dx, nullptr, s);
}

// ---------------------------------------------------------------- adapter gradients
size_t pact_lora_adapter_grad_workspace_size(int64_t M, int64_t N, int64_t K, int r) {
  if (M < 1 || N < 1 || K < 1 || r < 1 || r > 64) return 0;
  const int rp = rp_for(r);
  int64_t rps;
  const int64_t part_n = lora_ts_splits(M, N, rp, false, &rps) * N;
  const int64_t part_k = lora_ts_splits(M, K, rp, true, &rps) * K;
  return align256((size_t)rp * K * 2) + align256((size_t)N * rp * 2) +
         2 * align256((size_t)M * 2 * rp * 2) +
         align256((size_t)(part_n > part_k ? part_n : part_k) * rp * 4);
}

int pact_lora_adapter_grad(const pact_nvfp4* xq, const uint16_t* dy, const uint16_t* A,
                           const uint16_t* B, int r, float scale, int64_t N, float* dA, float* dB,
                           void* ws, size_t ws_bytes, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!xq) return fail(PACT_ERR_INVALID_ARG, "xq is required");
  const int64_t M = xq->rows, K = xq->cols;
  if ((rc = check_gemm_dims(M, N, K, r))) return rc;
  if ((rc = check_nvfp4(xq, "xq", M, K, 16))) return rc;
  if (!dy || !A || !B || !dA || !dB)
    return fail(PACT_ERR_INVALID_ARG, "dy, A, B, dA and dB are required");
  if (!aligned(dy, 16) || !aligned(B, 16) || !aligned(A, 2) || !aligned(dA, 4) || !aligned(dB, 4))
    return fail(PACT_ERR_ALIGN, "dy and B must be 16-byte aligned");
  if (!ws || ws_bytes < pact_lora_adapter_grad_workspace_size(M, N, K, r) || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  const int rp = rp_for(r);
  char* p = (char*)ws;
  uint16_t* at = (uint16_t*)p;
  p += align256((size_t)rp * K * 2);
  uint16_t* bt = (uint16_t*)p;
  p += align256((size_t)N * rp * 2);
  uint16_t* t = (uint16_t*)p;
  p += align256((size_t)M * 2 * rp * 2);
  uint16_t* u = (uint16_t*)p;
  p += align256((size_t)M * 2 * rp * 2);
  float* part = (float*)p;
  cudaError_t e = launch_lora_adapter_grad((const uint8_t*)xq->codes, (const uint8_t*)xq->sf, xq->g,
                                           M, K, dy, N, A, B, r, rp, scale, dA, dB, at, bt, t, u,
                                           part, d->sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "adapter gradient launch");
}

// ---------------------------------------------------------------- fused nonlinear ops
size_t pact_rmsnorm_quant_workspace_size(int64_t, int64_t) { return 256; }

int pact_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t H, float eps,
                       pact_nvfp4* yq, float* rstd, void* ws, size_t ws_bytes,
                       pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!x || !gamma || !rstd) return fail(PACT_ERR_INVALID_ARG, "x, gamma and rstd are required");
  if (M < 1 || H < 64 || H % 64 || H > 16384)
    return fail(PACT_ERR_SHAPE, "need M >= 1, H %% 64 == 0, H <= 16384");
  if (pad_to(M, 128) * (H / 16) >= (int64_t)1 << 31)
    return fail(PACT_ERR_SHAPE, "tensor too large: pad128(M) * H / 16 must be < 2^31");
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(rstd, 4))
    return fail(PACT_ERR_ALIGN, "x and gamma must be 16-byte aligned");
  if ((rc = check_nvfp4(yq, "yq", M, H, 16))) return rc;
  if (!ws || ws_bytes < 256 || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  CUtensorMap tmx;
  if ((rc = make_map(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, H, M, 64, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B)))
    return rc;
  cudaError_t e = launch_rmsnorm_quant(tmx, x, gamma, M, H, eps, (uint8_t*)yq->codes, (uint8_t*)yq->sf,
                                       yq->g, rstd, (unsigned*)ws, d->status, d->sms,
                                       (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "rmsnorm launch");
}

size_t pact_silu_mul_quant_workspace_size(int64_t, int64_t) { return 256; }

int pact_silu_mul_quant(const uint16_t* gateup, int64_t M, int64_t I, const float* amax3_opt,
                        pact_nvfp4* hq, pact_nvfp4* gate_q, pact_nvfp4* up_q, void* ws,
                        size_t ws_bytes, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!gateup) return fail(PACT_ERR_INVALID_ARG, "gateup is null");
  if (M < 1 || I < 64 || I % 64) return fail(PACT_ERR_SHAPE, "need M >= 1 and I %% 64 == 0");
  if (pad_to(M, 128) * (I / 16) >= (int64_t)1 << 31)
    return fail(PACT_ERR_SHAPE, "tensor too large: pad128(M) * I / 16 must be < 2^31");
  if (!aligned(gateup, 16)) return fail(PACT_ERR_ALIGN, "gateup must be 16-byte aligned");
  if ((rc = check_nvfp4(hq, "hq", M, I, 16)) || (rc = check_nvfp4(gate_q, "gate_q", M, I, 16)) ||
      (rc = check_nvfp4(up_q, "up_q", M, I, 16)))
    return rc;
  if (!ws || ws_bytes < 256 || !aligned(ws, 256))
    return fail(PACT_ERR_INVALID_ARG, "workspace missing, too small or not 256-byte aligned");
  uint8_t* codes[3] = {(uint8_t*)hq->codes, (uint8_t*)gate_q->codes, (uint8_t*)up_q->codes};
  uint8_t* sf[3] = {(uint8_t*)hq->sf, (uint8_t*)gate_q->sf, (uint8_t*)up_q->sf};
  float* g[3] = {hq->g, gate_q->g, up_q->g};
  cudaError_t e = launch_silu_mul_quant(gateup, M, I, amax3_opt, codes, sf, g, (unsigned*)ws,
                                        d->sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "silu launch");
}

int pact_silu_mul_bwd(const pact_nvfp4* gate_q, const pact_nvfp4* up_q, const uint16_t* dh,
                      uint16_t* dgateup, float* out_amax_opt, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!gate_q || !up_q || !dh || !dgateup)
    return fail(PACT_ERR_INVALID_ARG, "gate_q, up_q, dh and dgateup are required");
  const int64_t M = gate_q->rows, I = gate_q->cols;
  if (M < 1 || I < 64 || I % 64) return fail(PACT_ERR_SHAPE, "need M >= 1 and I %% 64 == 0");
  if (pad_to(M, 128) * (I / 16) >= (int64_t)1 << 31)
    return fail(PACT_ERR_SHAPE, "tensor too large: pad128(M) * I / 16 must be < 2^31");
  if ((rc = check_nvfp4(gate_q, "gate_q", M, I, 16)) || (rc = check_nvfp4(up_q, "up_q", M, I, 16)))
    return rc;
  if (!aligned(dh, 16) || !aligned(dgateup, 16))
    return fail(PACT_ERR_ALIGN, "dh and dgateup must be 16-byte aligned");
  cudaError_t e = launch_silu_mul_bwd(
      (const uint8_t*)gate_q->codes, (const uint8_t*)gate_q->sf, gate_q->g,
      (const uint8_t*)up_q->codes, (const uint8_t*)up_q->sf, up_q->g, dh, M, I, dgateup,
      (unsigned*)out_amax_opt, d->sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "silu bwd launch");
}

int pact_rmsnorm_bwd(const pact_nvfp4* yq, const uint16_t* gamma, const float* rstd,
                     const uint16_t* dy, const uint16_t* dres_opt, uint16_t* dx,
                     float* out_amax_opt, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!yq || !gamma || !rstd || !dy || !dx)
    return fail(PACT_ERR_INVALID_ARG, "yq, gamma, rstd, dy and dx are required");
  const int64_t M = yq->rows, H = yq->cols;
  if (M < 1 || H < 64 || H % 64 || H > 16384)
    return fail(PACT_ERR_SHAPE, "need M >= 1, H %% 64 == 0, H <= 16384");
  if ((rc = check_nvfp4(yq, "yq", M, H, 16))) return rc;
  if (!aligned(gamma, 16) || !aligned(dy, 16) || !aligned(dx, 16) ||
      (dres_opt && !aligned(dres_opt, 16)) || (out_amax_opt && !aligned(out_amax_opt, 4)))
    return fail(PACT_ERR_ALIGN, "gamma, dy, dres and dx must be 16-byte aligned");
  cudaError_t e = launch_rmsnorm_bwd((const uint8_t*)yq->codes, (const uint8_t*)yq->sf, yq->g,
                                     gamma, rstd, dy, dres_opt, M, H, dx,
                                     (unsigned*)out_amax_opt, d->sms, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "rmsnorm bwd launch");
}

int pact_test_wait_timeout(uint32_t limit_us, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (limit_us == 0 || limit_us > 2000000)
    return fail(PACT_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  cudaError_t e = launch_wait_timeout((uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "wait-timeout launch");
}

int pact_test_bounds_check(pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  cudaError_t e = launch_bounds_check((cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "bounds-check launch");
}

int pact_test_pexp(const float* x, float* y, int64_t n, pact_stream_t stream) {
  DeviceInfo* d;
  int rc = device_info(&d);
  if (rc) return rc;
  if (!x || !y || n < 0) return fail(PACT_ERR_INVALID_ARG, "bad pexp arguments");
  if (n == 0) return PACT_OK;
  cudaError_t e = launch_pexp(x, y, n, (cudaStream_t)stream);
  return e == cudaSuccess ? PACT_OK : cuda_fail(e, "pexp launch");
}

}  // extern "C"
