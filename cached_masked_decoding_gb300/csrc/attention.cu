// Instantiations of the block-attention kernel (head_dim 64/128, 2 or 4 query
// warps, 64-key tiles in bf16 or 32-key tiles that also carry the low halves).
#include "attention_tc.cuh"
#include "launch.h"

namespace dllm {

template <int HD, int WQ, int KT, bool LO = true>
static cudaError_t go_attn(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, dim3 grid,
                           cudaStream_t st, bool pdl) {
  const cudaError_t e = smem_attrs_once(reinterpret_cast<const void*>(attn_kernel<HD, WQ, KT, LO>),
                                        AttnCfg<HD, KT, LO>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_ex(attn_kernel<HD, WQ, KT, LO>, grid, dim3(128), AttnCfg<HD, KT, LO>::SMEM_BYTES, st, pdl, tk, tv,
                   p);
}

// 32-key tiles: with the low halves (split precision) or without (bf16, a
// smaller CTA, four per SM)
template <int HD, int WQ>
static cudaError_t go_attn32(const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p, dim3 grid,
                             cudaStream_t st, bool pdl) {
  return p.kv_lo ? go_attn<HD, WQ, 32, true>(tk, tv, p, grid, st, pdl)
                 : go_attn<HD, WQ, 32, false>(tk, tv, p, grid, st, pdl);
}

cudaError_t launch_attention(int hd, int wq, int kt, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnParams& p, dim3 grid, cudaStream_t st, bool pdl) {
  if (kt == 64 && p.kv_lo) return cudaErrorInvalidValue;   // 64-key tiles have no room for the low halves
  if (hd == 64 && wq == 2) return kt == 32 ? go_attn32<64, 2>(tk, tv, p, grid, st, pdl)
                                           : go_attn<64, 2, 64>(tk, tv, p, grid, st, pdl);
  if (hd == 64 && wq == 4) return kt == 32 ? go_attn32<64, 4>(tk, tv, p, grid, st, pdl)
                                           : go_attn<64, 4, 64>(tk, tv, p, grid, st, pdl);
  if (hd == 128 && wq == 2) return kt == 32 ? go_attn32<128, 2>(tk, tv, p, grid, st, pdl)
                                            : go_attn<128, 2, 64>(tk, tv, p, grid, st, pdl);
  if (hd == 128 && wq == 4) return kt == 32 ? go_attn32<128, 4>(tk, tv, p, grid, st, pdl)
                                            : go_attn<128, 4, 64>(tk, tv, p, grid, st, pdl);
  return cudaErrorInvalidValue;
}

template <int HD>
static cudaError_t go_attn_tc(const CUtensorMap& tq, const CUtensorMap& tqlo, const CUtensorMap& tk,
                              const CUtensorMap& tv, const AttnParams& p, dim3 grid, cudaStream_t st, bool pdl) {
  const cudaError_t e = smem_attrs_once(reinterpret_cast<const void*>(attn_tc_kernel<HD>), AttnTcCfg<HD>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_ex(attn_tc_kernel<HD>, grid, dim3(192), AttnTcCfg<HD>::SMEM_BYTES, st, pdl, tq, tqlo, tk, tv, p);
}

cudaError_t launch_attention_tc(int hd, const CUtensorMap& tq, const CUtensorMap& tqlo, const CUtensorMap& tk,
                                const CUtensorMap& tv, const AttnParams& p, dim3 grid, cudaStream_t st, bool pdl) {
  if (hd == 64) return go_attn_tc<64>(tq, tqlo, tk, tv, p, grid, st, pdl);
  if (hd == 128) return go_attn_tc<128>(tq, tqlo, tk, tv, p, grid, st, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace dllm
