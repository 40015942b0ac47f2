// Instantiations of the persistent DualCache step kernel for head_dim 64.
#include "launch.h"
#include "step_kernel.cuh"

namespace dllm {

template <int BN>
static cudaError_t go_step_64(const StepArgs& a, int grid, cudaStream_t st) {
  const cudaError_t e = smem_attrs_once(reinterpret_cast<const void*>(step_kernel<BN, 64>),
                                        StepCfg<BN, 64>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = StepCfg<BN, 64>::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<BN, 64>, a);
}

cudaError_t launch_step_hd64(int bn, const StepArgs& a, int grid, cudaStream_t st) {
  switch (bn) {
    case 32: return go_step_64<32>(a, grid, st);
    case 64: return go_step_64<64>(a, grid, st);
    case 128: return go_step_64<128>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dllm
