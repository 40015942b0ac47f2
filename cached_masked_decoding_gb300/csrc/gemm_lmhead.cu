// Instantiations of the tensor-core GEMM with the lmhead epilogue.
#include "launch.h"

DLLM_GEMM_LAUNCHER(lmhead, GEMM_LMHEAD)
