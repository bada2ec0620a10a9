// LoRA linear forward for callers that cannot allocate device memory.
//
// pact_lora_linear_fwd needs a caller-provided workspace for its intermediate
// LoRA operands.  Some callers have no way to provide one: a plugin whose host
// framework hands it only inputs and outputs, code that runs while a stream is
// being captured into a CUDA graph (cudaMalloc is not allowed there), or a
// runtime with a fixed device-memory budget where a cudaMalloc on the hot path
// would synchronise the device.  This entry point runs the same computation with
// its scratch in a fixed array that is part of the library image: every GPU that
// loads the library holds the array until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/pact.h"
#include "kernels.h"

namespace {

// Fixed scratch for pact_lora_linear_fwd_noalloc (PACT_NOALLOC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PACT_NOALLOC_SCRATCH_BYTES];

struct ScratchAddr {
  bool ready = false;
  void* ptr = nullptr;
};
ScratchAddr g_addr[64];
std::mutex g_addr_mu;

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pact::report_error(PACT_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return pact::report_error(PACT_ERR_INVALID_ARG, "device index");
  std::lock_guard<std::mutex> lk(g_addr_mu);
  if (!g_addr[dev].ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return pact::report_error(PACT_ERR_CUDA, "cudaGetSymbolAddress of the no-alloc scratch failed");
    g_addr[dev].ptr = p;
    g_addr[dev].ready = true;
  }
  *out = g_addr[dev].ptr;
  return PACT_OK;
}

}  // namespace

extern "C" {

size_t pact_lora_linear_fwd_noalloc_max_scratch(void) { return PACT_NOALLOC_SCRATCH_BYTES; }

int pact_lora_linear_fwd_noalloc(const pact_nvfp4* xq, const pact_nvfp4* w_fwd,
                                 const uint16_t* A, const uint16_t* B, int r, float scale,
                                 const uint16_t* residual_opt, uint16_t* y, float* out_amax_opt,
                                 pact_stream_t stream) {
  if (!xq || !w_fwd) return pact::report_error(PACT_ERR_INVALID_ARG, "xq and w_fwd are required");
  const size_t need = pact_lora_linear_fwd_workspace_size(xq->rows, w_fwd->rows, xq->cols, r);
  if (need == 0) return pact::report_error(PACT_ERR_INVALID_ARG, "bad shape or rank (1 <= r <= 64)");
  if (need > PACT_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "this call needs %zu bytes of scratch; the no-alloc entry point has a fixed %zu "
             "(use pact_lora_linear_fwd with a workspace)",
             need, (size_t)PACT_NOALLOC_SCRATCH_BYTES);
    return pact::report_error(PACT_ERR_SHAPE, msg);
  }
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc != PACT_OK) return rc;
  // The forward writes every scratch byte it later reads (both LoRA operands,
  // zero padding included) before reading it, so nothing needs clearing here.
  return pact_lora_linear_fwd(xq, w_fwd, A, B, r, scale, residual_opt, y, out_amax_opt, ws,
                              PACT_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
