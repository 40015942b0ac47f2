// Instantiations of the tensor-core GEMM with the plain epilogue.
#include "launch.h"

DLLM_GEMM_LAUNCHER(plain, GEMM_PLAIN)
