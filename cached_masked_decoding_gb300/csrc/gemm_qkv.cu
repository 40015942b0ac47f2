// Instantiations of the tensor-core GEMM with the qkv epilogue.
#include "launch.h"

DLLM_GEMM_LAUNCHER(qkv, GEMM_QKV)
