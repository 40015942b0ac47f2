// Instantiations of the tensor-core GEMM with the resid epilogue.
#include "launch.h"

DLLM_GEMM_LAUNCHER(resid, GEMM_RESID)
