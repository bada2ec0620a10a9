// The device status word: its bits, and the debug build's checks that set them.
//
// Kernels record errors here instead of trapping; pact_check_status reads and
// clears the word.  Debug builds (PACT_DEBUG: the whole library as the one
// translation unit debug_all.cu) add two kinds of check, which release builds
// compile away:
//   - the index arithmetic of the kernels' hand-computed stores against the buffer
//     extents (PACT_IN): a failed check records PACT_DEV_BOUNDS and the store is
//     skipped, so an out-of-bounds index shows up in pact_check_status instead of
//     corrupting memory;
//   - NaN in the values a quantisation, statistic or output amax reads
//     (PACT_NAN_*): inputs are finite by contract, and a NaN records PACT_DEV_NAN
//     while the values are used as they are.
#pragma once

#include <stdint.h>

namespace pact {

enum : unsigned {
  PACT_DEV_TIMEOUT = 1u,
  PACT_DEV_BOUNDS = 1u << 1,  // a bounds check of the debug build failed
  PACT_DEV_NAN = 1u << 2,     // the debug build saw a NaN value
  PACT_DEV_ROLE_TMA = 1u << 8,
  PACT_DEV_ROLE_MMA = 1u << 9,
  PACT_DEV_ROLE_EPI = 1u << 10,
  PACT_DEV_ROLE_SF = 1u << 11,
};

#ifdef PACT_DEBUG
// the status word itself (the debug build is a single unit; release builds define
// it in gemm.cu)
__device__ unsigned g_pact_status;
__device__ __forceinline__ bool in_bounds(bool ok) {
  if (!ok) atomicOr(&g_pact_status, PACT_DEV_BOUNDS);
  return ok;
}
// two BF16 values packed in a word: NaN is exponent all ones with a nonzero mantissa
__device__ __forceinline__ void nan_check_bf16x2(uint32_t w) {
  if ((w & 0x7FFFu) > 0x7F80u || ((w >> 16) & 0x7FFFu) > 0x7F80u)
    atomicOr(&g_pact_status, PACT_DEV_NAN);
}
__device__ __forceinline__ void nan_check_f32(float v) {
  if (v != v) atomicOr(&g_pact_status, PACT_DEV_NAN);
}
#define PACT_IN(cond) ::pact::in_bounds(cond)
#define PACT_NAN_BF16X2(w) ::pact::nan_check_bf16x2(w)
#define PACT_NAN_F32(v) ::pact::nan_check_f32(v)
#else
#define PACT_IN(cond) true
#define PACT_NAN_BF16X2(w) ((void)0)
#define PACT_NAN_F32(v) ((void)0)
#endif

}  // namespace pact
