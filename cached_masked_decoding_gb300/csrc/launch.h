// Host-side launchers of the kernel templates (one translation unit per GEMM
// epilogue kind so the build compiles them in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <utility>

#include "attention.cuh"
#include "gemm.cuh"
#include "step_kernel.cuh"

namespace dllm {

// A kernel's dynamic shared-memory limit and carveout are attributes of the
// function on the current device: set them once per (kernel, device), under a
// lock, so that host threads and devices do not race or miss them.
inline cudaError_t smem_attrs_once(const void* kernel, int smem_bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  // every kernel of the step asks for the same L1/shared split, so an SM
  // never has to drain and reconfigure between them
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  done.insert({kernel, dev});
  return cudaSuccess;
}

// Launch with programmatic dependent launch allowed (pdl) on stream st.
template <typename Kern, typename... Args>
inline cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_gemm_plain(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,
                              cudaStream_t st, bool pdl);
cudaError_t launch_gemm_qkv(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,
                            cudaStream_t st, bool pdl);
cudaError_t launch_gemm_resid(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,
                              cudaStream_t st, bool pdl);
cudaError_t launch_gemm_swiglu(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,
                               cudaStream_t st, bool pdl);
cudaError_t launch_gemm_lmhead(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,
                               cudaStream_t st, bool pdl);

inline cudaError_t launch_gemm(int kind, int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p,
                               int grid, cudaStream_t st, bool pdl) {
  switch (kind) {
    case GEMM_PLAIN: return launch_gemm_plain(bn, a, b, blo, p, grid, st, pdl);
    case GEMM_QKV: return launch_gemm_qkv(bn, a, b, blo, p, grid, st, pdl);
    case GEMM_RESID: return launch_gemm_resid(bn, a, b, blo, p, grid, st, pdl);
    case GEMM_SWIGLU: return launch_gemm_swiglu(bn, a, b, blo, p, grid, st, pdl);
    case GEMM_LMHEAD: return launch_gemm_lmhead(bn, a, b, blo, p, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_step_hd64(int bn, const StepArgs& a, int grid, cudaStream_t st);
cudaError_t launch_step_hd128(int bn, const StepArgs& a, int grid, cudaStream_t st);

// kt: keys per shared-memory tile, 64 (bf16 K/V) or 32 (also with low halves,
// p.kv_lo); the tensor maps' key box must match.
cudaError_t launch_attention(int hd, int wq, int kt, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnParams& p, dim3 grid, cudaStream_t st, bool pdl);

// Tensor-core attention over 128-query tiles (attention_tc.cuh): grid
// (ceil(R/128), H, b); tq/tqlo: 128-row maps over q and q_lo (tqlo unused
// unless p.kv_lo); tk/tv: K/V maps with 64-key boxes.  hd in {64, 128}.
cudaError_t launch_attention_tc(int hd, const CUtensorMap& tq, const CUtensorMap& tqlo, const CUtensorMap& tk,
                                const CUtensorMap& tv, const AttnParams& p, dim3 grid, cudaStream_t st, bool pdl);

}  // namespace dllm

// Instantiate launch_gemm_<name> for the four activation-tile widths.
#define DLLM_GEMM_LAUNCHER(NAME, KIND)                                                                            \
  namespace dllm {                                                                                              \
  template <int BN>                                                                                             \
  static cudaError_t go_##NAME(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p, int grid,       \
                               cudaStream_t st, bool pdl) {                                                     \
    const cudaError_t e = smem_attrs_once(reinterpret_cast<const void*>(gemm_kernel<BN, KIND>),                 \
                                          GemmCfg<BN>::SMEM_BYTES);                                             \
    if (e != cudaSuccess) return e;                                                                             \
    return launch_ex(gemm_kernel<BN, KIND>, dim3(grid), dim3(192), GemmCfg<BN>::SMEM_BYTES, st, pdl, a, b, blo, p);  \
  }                                                                                                             \
  cudaError_t launch_gemm_##NAME(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& blo, const GemmParams& p,       \
                                 int grid, cudaStream_t st, bool pdl) {                                         \
    switch (bn) {                                                                                               \
      case 32: return go_##NAME<32>(a, b, blo, p, grid, st, pdl);                                                    \
      case 64: return go_##NAME<64>(a, b, blo, p, grid, st, pdl);                                                    \
      case 128: return go_##NAME<128>(a, b, blo, p, grid, st, pdl);                                                  \
      case 256: return go_##NAME<256>(a, b, blo, p, grid, st, pdl);                                                  \
      default: return cudaErrorInvalidValue;                                                                    \
    }                                                                                                           \
  }                                                                                                             \
  }
