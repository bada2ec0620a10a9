// The whole library as one translation unit, for the debug build (-DPACT_DEBUG):
// the bounds checks of every kernel record failures in the one device status word
// defined in gemm.cu, which needs every kernel in the same unit (the release build
// compiles the files separately and the checks away).
#include "api.cu"
#include "quant.cu"
#include "gemm.cu"
#include "lora.cu"
#include "norm_act.cu"
#include "noalloc.cu"
