// Instantiations of the tensor-core GEMM with the swiglu epilogue.
#include "launch.h"

DLLM_GEMM_LAUNCHER(swiglu, GEMM_SWIGLU)
