// Host side of libdllm: models, decoding states, the denoise-step pipeline and
// the C ABI of include/dllm.h.
//
// One denoise step (Algorithm 1, steps 5-10 of the Fast-dLLM notes) is a chain
// of kernels on the state's stream, each launched with programmatic dependent
// launch so the next weight stream starts while the previous kernel drains:
//   embed -> per layer [QKV+RoPE+K/V write, attention, O-proj+residual+norm,
//   gate/up+SwiGLU, down+residual+norm] -> LM head + softmax statistics ->
//   merge + select/commit.
// The only device->host traffic of a step is the committed count per sequence.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <array>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/dllm.h"
#include "launch.h"
#include "small_kernels.cuh"

using namespace dllm;

// ====================================================================== errors
namespace {

thread_local char g_err[2048] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

#define CK(call)                                                                                   \
  do {                                                                                             \
    cudaError_t e_ = (call);                                                                       \
    if (e_ != cudaSuccess) {                                                                       \
      set_error("%s:%d %s: %s", __FILE__, __LINE__, #call, cudaGetErrorString(e_));                \
      return DLLM_ECUDA;                                                                           \
    }                                                                                              \
  } while (0)

#define CKS(expr)                         \
  do {                                    \
    dllm_status s_ = (expr);              \
    if (s_ != DLLM_OK) return s_;         \
  } while (0)

// Host-side fault injection for tests: DLLM_FAULT=alloc makes device
// allocations fail, DLLM_FAULT=io makes weight-file reads fail.
bool fault(const char* what) {
  const char* f = std::getenv("DLLM_FAULT");
  return f && std::strcmp(f, what) == 0;
}

dllm_status dev_alloc(void** p, size_t bytes) {
  *p = nullptr;
  if (fault("alloc")) {
    set_error("device allocation of %zu bytes refused (DLLM_FAULT=alloc)", bytes);
    return DLLM_ENOMEM;
  }
  if (bytes == 0) bytes = 256;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    set_error("cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? DLLM_ENOMEM : DLLM_ECUDA;
  }
  return DLLM_OK;
}

// ====================================================================== tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [rows][inner] matrix, box [box_rows][64], 128-byte swizzle.
dllm_status map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return DLLM_ECUDA;
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled(2d, inner=%llu rows=%llu box_rows=%u) failed: %d",
              (unsigned long long)inner, (unsigned long long)rows, box_rows, (int)r);
    return DLLM_ECUDA;
  }
  return DLLM_OK;
}

// Keys per shared-memory tile of the state's attention (32: room for the low
// halves of K and V next to them).
constexpr int kStateAttnKT = 32;

// 3-D bf16 map over [planes][T][hd] (K or V planes of the cache), box [1][keys][64].
dllm_status map_kv(CUtensorMap* m, const void* base, uint64_t hd, uint64_t T, uint64_t planes, uint32_t keys) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return DLLM_ECUDA;
  }
  cuuint64_t dims[3] = {hd, T, planes};
  cuuint64_t strides[2] = {hd * 2, T * hd * 2};
  cuuint32_t box[3] = {64, keys, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled(3d kv) failed: %d", (int)r);
    return DLLM_ECUDA;
  }
  return DLLM_OK;
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }
int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

int pick_bn(int n, bool split = false) {
  if (n <= 32) return 32;
  if (n <= 64) return 64;
  if (n <= 128 || split) return 128;
  return 256;
}

int device_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

struct AttnPlan {
  int wq, q_tiles, splits, kps;
  long long n_whole = 0;   // tensor-core plan: leading query tiles run unsplit (whole waves)
};

AttnPlan plan_attention(int b, int H, int R, int T, int sms) {
  AttnPlan a;
  a.wq = R <= 32 ? 2 : 4;
  const int QT = 16 * a.wq;
  a.q_tiles = ceil_div(R, QT);
  const long long items = (long long)b * H * a.q_tiles;
  const int max_splits = std::max(1, ceil_div(T, 64));
  // about two CTAs per SM; at most 32 splits (the merge keeps QT x splits
  // weights in shared memory)
  int splits = 1;
  const long long target = 2LL * sms;
  if (items < target) splits = (int)std::min<long long>(max_splits, (target + items - 1) / items);
  splits = std::min(splits, 32);
  a.kps = round_up(ceil_div(T, splits), 64);
  a.splits = ceil_div(T, a.kps);
  return a;
}

// Attention plan of the persistent step: at most one work item per CTA.
AttnPlan plan_attention_persistent(int b, int H, int R, int T, int ctas) {
  AttnPlan a;
  a.wq = 2;
  a.q_tiles = ceil_div(R, 32);
  const long long base = (long long)b * H * a.q_tiles;
  const int max_splits = std::max(1, ceil_div(T, 64));
  int splits = (int)std::max<long long>(1, std::min<long long>(max_splits, ctas / std::max<long long>(base, 1)));
  splits = std::min(splits, 32);
  a.kps = round_up(ceil_div(T, splits), 64);
  a.splits = ceil_div(T, a.kps);
  return a;
}

// Persistent step kinds (see step_rows) and the shape of one phase list.
enum StepKind : int { SK_DUAL = 0, SK_COMMIT = 1, SK_KINDS = 2 };
struct StepShape {
  int bn = 0;     // activation tile rows (the kernel template); 0: no list
  int rows = 0;   // rows per sequence
  int row0 = 0;   // position of the first row
  AttnPlan ap = {};
};

// Query rows per sequence from which attention runs on the tensor cores
// (128-query tiles); fewer rows use the key-split kernel.
constexpr int kAttnTcMinRows = 65;

// Plan of the tensor-core attention (128-query tiles, 64-key tiles): key
// splits when the query tiles fill the GPU's SMs unevenly.  One CTA per SM;
// the cost of a round of CTAs is taken as the key tiles a CTA walks plus
// fixed work: one tile's worth unsplit, four with a partial and its merge
// (measured on GB300: the 8B refresh's 192 query tiles took 65.7 us unsplit
// and 73.9 us with every tile in two splits; a PrefixCache step's 64 tiles
// 33.8 and 29.0 us).  Two shapes are weighed: every query tile in s splits,
// or whole waves of unsplit tiles followed by the remaining tiles in s
// splits.  Splits are taken only when they promise at least a tenth less
// time; at most 8 (the merge keeps 128 x splits weights in shared memory).
AttnPlan plan_attention_tc(int b, int H, int R, int T, int sms) {
  AttnPlan a;
  a.wq = 8;
  a.q_tiles = ceil_div(R, 128);
  const long long items = (long long)b * H * a.q_tiles;
  const int kt = std::max(1, ceil_div(T, 64));
  auto rounds = [&](long long n) { return (n + sms - 1) / sms; };
  auto per = [&](int sp) { return (long long)ceil_div(kt, sp) + (sp > 1 ? 4 : 1); };
  const long long unsplit = rounds(items) * per(1);
  const long long whole = (items / sms) * sms, rem = items - whole;
  long long best = unsplit, best_whole = 0;
  int best_sp = 1;
  for (int sp = 2; sp <= 8 && sp <= kt; ++sp) {
    const long long uniform = rounds(items * sp) * per(sp);
    if (uniform < best) {
      best = uniform;
      best_sp = sp;
      best_whole = 0;
    }
    if (whole > 0 && rem > 0) {
      const long long hybrid = (whole / sms) * per(1) + rounds(rem * sp) * per(sp);
      if (hybrid < best) {
        best = hybrid;
        best_sp = sp;
        best_whole = whole;
      }
    }
  }
  if (best_sp > 1 && 10 * best > 9 * unsplit) {
    best_sp = 1;
    best_whole = 0;
  }
  a.kps = ceil_div(kt, best_sp) * 64;
  a.splits = ceil_div(T, a.kps);
  a.n_whole = a.splits > 1 ? best_whole : 0;
  return a;
}

// CTAs of a tensor-core plan and the query tiles that go through the merge.
long long tc_ctas(const AttnPlan& a, long long items) { return a.n_whole + (items - a.n_whole) * a.splits; }
long long tc_split_items(const AttnPlan& a, long long items) { return a.splits > 1 ? items - a.n_whole : 0; }

}  // namespace

// ====================================================================== model
struct LayerW {
  uint16_t *attn_norm, *wqkv, *wo, *ffn_norm, *wgu, *wd;
  CUtensorMap tm_qkv, tm_o, tm_gu, tm_d;
};

struct dllm_model {
  dllm_config cfg;
  int F_pad;
  int sms;
  void* arena = nullptr;
  size_t arena_bytes = 0;
  uint16_t *embed = nullptr, *final_norm = nullptr, *lm = nullptr;
  std::vector<LayerW> layers;
  CUtensorMap tm_lm;
};

namespace {

dllm_status check_config(const dllm_config* c) {
  if (!c) {
    set_error("config is NULL");
    return DLLM_EINVAL;
  }
  if (c->n_layers < 1 || c->d_model < 128 || c->d_model % 128 != 0 || c->n_heads < 1 ||
      (c->head_dim != 64 && c->head_dim != 128) || c->n_heads * c->head_dim != c->d_model || c->d_ffn < 1 ||
      c->vocab < 2 || c->d_model > 8192 || !(c->rope_theta > 0) || !(c->norm_eps >= 0)) {
    set_error("unsupported config: layers=%d d=%d heads=%d head_dim=%d ffn=%d vocab=%d (need d %% 128 == 0, "
              "head_dim 64|128, heads*head_dim == d, d <= 8192)",
              c->n_layers, c->d_model, c->n_heads, c->head_dim, c->d_ffn, c->vocab);
    return DLLM_EINVAL;
  }
  return DLLM_OK;
}

}  // namespace

extern "C" dllm_status dllm_model_create(const dllm_config* cfg, dllm_model** out) {
  if (!out) {
    set_error("out is NULL");
    return DLLM_EINVAL;
  }
  *out = nullptr;
  CKS(check_config(cfg));
  dllm_model* m = new dllm_model();
  m->cfg = *cfg;
  m->F_pad = round_up(cfg->d_ffn, 64);
  m->sms = device_sms();
  const size_t d = cfg->d_model, F = m->F_pad, V = cfg->vocab, L = cfg->n_layers;
  auto al = [](size_t bytes) { return (bytes + 1023) / 1024 * 1024; };
  const size_t per_layer = al(d * 2) * 2 + al(3 * d * d * 2) + al(d * d * 2) + al(2 * F * d * 2) + al(d * F * 2);
  m->arena_bytes = al((V + 1) * d * 2) + al(d * 2) + al(V * d * 2) + L * per_layer;
  dllm_status st = dev_alloc(&m->arena, m->arena_bytes);
  if (st != DLLM_OK) {
    delete m;
    return st;
  }
  cudaError_t e = cudaMemset(m->arena, 0, m->arena_bytes);
  if (e != cudaSuccess) {
    cudaFree(m->arena);
    delete m;
    set_error("cudaMemset of the weight arena failed: %s", cudaGetErrorString(e));
    return DLLM_ECUDA;
  }
  uint8_t* p = static_cast<uint8_t*>(m->arena);
  auto take = [&](size_t bytes) {
    uint16_t* r = reinterpret_cast<uint16_t*>(p);
    p += al(bytes);
    return r;
  };
  m->embed = take((V + 1) * d * 2);
  m->final_norm = take(d * 2);
  m->lm = take(V * d * 2);
  m->layers.resize(L);
  for (size_t l = 0; l < L; ++l) {
    LayerW& w = m->layers[l];
    w.attn_norm = take(d * 2);
    w.ffn_norm = take(d * 2);
    w.wqkv = take(3 * d * d * 2);
    w.wo = take(d * d * 2);
    w.wgu = take(2 * F * d * 2);
    w.wd = take(d * F * 2);
    if ((st = map_2d(&w.tm_qkv, w.wqkv, d, 3 * d, 128)) != DLLM_OK ||
        (st = map_2d(&w.tm_o, w.wo, d, d, 128)) != DLLM_OK ||
        (st = map_2d(&w.tm_gu, w.wgu, d, 2 * F, 128)) != DLLM_OK ||
        (st = map_2d(&w.tm_d, w.wd, F, d, 128)) != DLLM_OK) {
      cudaFree(m->arena);
      delete m;
      return st;
    }
  }
  if ((st = map_2d(&m->tm_lm, m->lm, d, V, 128)) != DLLM_OK) {
    cudaFree(m->arena);
    delete m;
    return st;
  }
  *out = m;
  return DLLM_OK;
}

extern "C" void dllm_free_model(dllm_model* m) {
  if (!m) return;
  if (m->arena) cudaFree(m->arena);
  delete m;
}

extern "C" dllm_status dllm_model_config(const dllm_model* m, dllm_config* cfg) {
  if (!m || !cfg) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  *cfg = m->cfg;
  return DLLM_OK;
}

namespace {

int64_t tensor_count(const dllm_config& c, int t) {
  const int64_t d = c.d_model, F = c.d_ffn, V = c.vocab;
  switch (t) {
    case DLLM_T_EMBED: return (V + 1) * d;
    case DLLM_T_ATTN_NORM:
    case DLLM_T_FFN_NORM:
    case DLLM_T_FINAL_NORM: return d;
    case DLLM_T_WQ:
    case DLLM_T_WK:
    case DLLM_T_WV:
    case DLLM_T_WO: return d * d;
    case DLLM_T_WG:
    case DLLM_T_WU:
    case DLLM_T_WD: return F * d;
    case DLLM_T_LM_HEAD: return V * d;
    default: return -1;
  }
}

}  // namespace

extern "C" dllm_status dllm_model_set_tensor(dllm_model* m, int32_t tensor, int32_t layer, const uint16_t* src,
                                             int64_t count, int32_t src_on_device) {
  if (!m || !src) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  const dllm_config& c = m->cfg;
  const int64_t want = tensor_count(c, tensor);
  if (want < 0) {
    set_error("unknown tensor id %d", tensor);
    return DLLM_EINVAL;
  }
  const bool per_layer = tensor >= DLLM_T_ATTN_NORM && tensor <= DLLM_T_WD;
  if (per_layer && (layer < 0 || layer >= c.n_layers)) {
    set_error("layer %d out of range [0, %d)", layer, c.n_layers);
    return DLLM_EINVAL;
  }
  if (count != want) {
    set_error("tensor %d expects %lld values, got %lld", tensor, (long long)want, (long long)count);
    return DLLM_EINVAL;
  }
  const cudaMemcpyKind kind = src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  const size_t d = c.d_model, F = c.d_ffn, Fp = m->F_pad;
  LayerW* w = per_layer ? &m->layers[layer] : nullptr;
  switch (tensor) {
    case DLLM_T_EMBED: CK(cudaMemcpy(m->embed, src, count * 2, kind)); break;
    case DLLM_T_FINAL_NORM: CK(cudaMemcpy(m->final_norm, src, count * 2, kind)); break;
    case DLLM_T_LM_HEAD: CK(cudaMemcpy(m->lm, src, count * 2, kind)); break;
    case DLLM_T_ATTN_NORM: CK(cudaMemcpy(w->attn_norm, src, count * 2, kind)); break;
    case DLLM_T_FFN_NORM: CK(cudaMemcpy(w->ffn_norm, src, count * 2, kind)); break;
    case DLLM_T_WQ:
    case DLLM_T_WK:
    case DLLM_T_WV:
      CK(cudaMemcpy(w->wqkv + (size_t)(tensor - DLLM_T_WQ) * d * d, src, count * 2, kind));
      break;
    case DLLM_T_WO: CK(cudaMemcpy(w->wo, src, count * 2, kind)); break;
    case DLLM_T_WG:
    case DLLM_T_WU: {
      // gate/up interleaved in 64-row groups: rows [128i, 128i+64) gate, [128i+64, 128i+128) up
      const size_t off = tensor == DLLM_T_WU ? 64 : 0;
      for (size_t f0 = 0; f0 < F; f0 += 64) {
        const size_t rows = std::min<size_t>(64, F - f0);
        CK(cudaMemcpy(w->wgu + ((f0 / 64) * 128 + off) * d, src + f0 * d, rows * d * 2, kind));
      }
      break;
    }
    case DLLM_T_WD:
      CK(cudaMemcpy2D(w->wd, Fp * 2, src, F * 2, F * 2, d, kind));
      break;
    default: set_error("unknown tensor"); return DLLM_EINVAL;
  }
  return DLLM_OK;
}

extern "C" dllm_status dllm_load(const char* path, dllm_model** out) {
  if (!path || !out) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  *out = nullptr;
  if (fault("io")) {
    set_error("weight file read refused (DLLM_FAULT=io)");
    return DLLM_EIO;
  }
  FILE* fh = std::fopen(path, "rb");
  if (!fh) {
    set_error("cannot open %s", path);
    return DLLM_EIO;
  }
  char magic[8];
  int32_t hdr[6];
  float flt[2];
  if (std::fread(magic, 1, 8, fh) != 8 || std::memcmp(magic, "DLLMW001", 8) != 0 ||
      std::fread(hdr, 4, 6, fh) != 6 || std::fread(flt, 4, 2, fh) != 2) {
    std::fclose(fh);
    set_error("%s: bad header", path);
    return DLLM_EIO;
  }
  dllm_config c{hdr[0], hdr[1], hdr[2], hdr[3], hdr[4], hdr[5], flt[0], flt[1]};
  dllm_model* m = nullptr;
  dllm_status st = dllm_model_create(&c, &m);
  if (st != DLLM_OK) {
    std::fclose(fh);
    return st;
  }
  std::vector<int> order;
  std::vector<int> layers;
  order.push_back(DLLM_T_EMBED);
  layers.push_back(0);
  const int per[] = {DLLM_T_ATTN_NORM, DLLM_T_WQ, DLLM_T_WK, DLLM_T_WV, DLLM_T_WO,
                     DLLM_T_FFN_NORM, DLLM_T_WG, DLLM_T_WU, DLLM_T_WD};
  for (int l = 0; l < c.n_layers; ++l)
    for (int t : per) {
      order.push_back(t);
      layers.push_back(l);
    }
  order.push_back(DLLM_T_FINAL_NORM);
  layers.push_back(0);
  order.push_back(DLLM_T_LM_HEAD);
  layers.push_back(0);
  std::vector<uint16_t> buf;
  for (size_t i = 0; i < order.size(); ++i) {
    const int64_t n = tensor_count(c, order[i]);
    buf.resize(n);
    if ((int64_t)std::fread(buf.data(), 2, n, fh) != n) {
      std::fclose(fh);
      dllm_free_model(m);
      set_error("%s: file ends inside tensor %d (layer %d)", path, order[i], layers[i]);
      return DLLM_EIO;
    }
    st = dllm_model_set_tensor(m, order[i], layers[i], buf.data(), n, 0);
    if (st != DLLM_OK) {
      std::fclose(fh);
      dllm_free_model(m);
      return st;
    }
  }
  std::fclose(fh);
  *out = m;
  return DLLM_OK;
}

// ====================================================================== state
// kernel classes of a denoise step; a refresh's launches use class + KC_REFRESH
enum KClass { KC_EMBED = 0, KC_QKV, KC_ATTN, KC_O, KC_GU, KC_D, KC_LM, KC_MERGE, KC_REFRESH = 8, KC_PSTEP = 14, KC_N = 16 };

struct dllm_state {
  dllm_model* m = nullptr;
  int b = 0, P = 0, gen = 0, B = 0, T = 0, n_blocks = 0;
  cudaStream_t st = nullptr;
  bool own_stream = false;
  void* arena = nullptr;
  int32_t* x = nullptr;
  uint16_t* kv = nullptr;
  float* h = nullptr;
  uint16_t* xn = nullptr;
  uint16_t* xn_lo = nullptr;
  float* ss = nullptr;
  uint16_t* q = nullptr;
  uint16_t* q_lo = nullptr;
  uint16_t* ao = nullptr;
  uint16_t* ao_lo = nullptr;
  uint16_t* act = nullptr;
  uint16_t* act_lo = nullptr;
  uint16_t* xf = nullptr;
  uint16_t* xf_lo = nullptr;
  bool split = true;              // activations as hi/lo bf16 pairs
  float* ssf = nullptr;
  float *st_m = nullptr, *st_s = nullptr;
  int* st_a = nullptr;
  float* conf = nullptr;
  int32_t* arg = nullptr;
  int32_t* count_err = nullptr;   // [b] counts, then the error word
  int* seq_done = nullptr;        // [b] merge arrival counters
  float* gemm_ws = nullptr;
  int* gemm_cnt = nullptr;
  float* attn_o = nullptr;
  size_t attn_o_floats = 0;   // attention merge workspace (partials and (m, l)), floats
  size_t attn_cnt_n = 0;      // merge counters
  float* attn_ml = nullptr;
  int* attn_cnt = nullptr;
  float2* rope = nullptr;
  int32_t* host_ce = nullptr;     // pinned copies of count_err: two slots of b + 1 (steps in flight at once)
  CUtensorMap tm_kv;
  std::map<std::tuple<const void*, int, int, int>, CUtensorMap> act_maps;
  std::map<const void*, CUtensorMap> kv64_maps;   // 64-key K/V maps of the tensor-core attention, per cache buffer
  std::vector<int32_t> prompts;   // host copy of the prompt part
  std::vector<int32_t> remaining; // [b][n_blocks] MASK count per block
  // last step
  int last_row0 = 0, last_R = 0, last_blk = 0;
  // trace
  bool trace = false;
  float* trace_buf = nullptr;
  // per-kernel timing
  bool timing = false;
  bool fused_fwd = false;   // a no-cache step standing in for a refresh and its step: timed as refresh kernels
  bool fuse_refresh = true; // dllm_run fuses refreshes and commit forwards with the step after them
  std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> pending;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_next = 0;
  double kt_ms[KC_N] = {0};
  long long kt_n[KC_N] = {0};
  double kt_bytes[KC_N] = {0};
  cudaEvent_t ev_a = nullptr, ev_b = nullptr;   // step or refresh timing (host slot 0)
  cudaEvent_t ev_c = nullptr, ev_d = nullptr;   // step timing (host slot 1)
  cudaEvent_t ev_done[2] = {nullptr, nullptr};  // a host slot's counts have landed
  bool run_ahead = true;          // dllm_run launches a block's next step before reading the current one's commits
  long long launches = 0;         // kernels launched by this state
  // persistent DualCache step (one cooperative launch per step)
  bool persistent = true;
  bool step_built = false;
  bool step_split = true;
  int n_phases = 0;
  int map_kv = 0;
  StepPhase* d_phases = nullptr;  // [SK_KINDS][n_blocks][n_phases]
  std::vector<StepShape> step_shape;   // [SK_KINDS][n_blocks]
  CUtensorMap* d_maps = nullptr;
  // staleness diagnostics (allocated on first use)
  uint16_t* kv_fresh = nullptr;   // K/V of a full forward over the current canvas, the cache's layout
  CUtensorMap tm_kv_fresh;
  int32_t* x_save = nullptr;      // canvas saved around the diagnostic forwards
  float* row_cos = nullptr;       // [L][K|V][b][H][T] cosine of cached and fresh rows
  int* d_flags = nullptr;         // dataflow flags of the persistent step, zeroed per launch
  int n_flags = 0;
  // weight tiles a CTA loads for a phase before its inputs are ready: 4 of
  // the 8 ring slots (8B workload, batch 1: 4.004 ms per step against 4.030
  // with the whole ring; fewer loads queued when the phase tail runs)
  int step_prefetch = 4;
  bool block_causal = false;                  // DLLM_MASK_BLOCK_CAUSAL
  unsigned long long* d_timeline = nullptr;   // persistent-step phase timeline (diagnostics)
  bool timeline = false;
  dllm_run_hook hook = nullptr;               // observer of dllm_run's events (nullable)
  void* hook_user = nullptr;
};

namespace {

dllm_status state_free_device(dllm_state* s) {
  if (s->arena) cudaFree(s->arena);
  if (s->gemm_ws) cudaFree(s->gemm_ws);
  if (s->trace_buf) cudaFree(s->trace_buf);
  if (s->d_phases) cudaFree(s->d_phases);
  if (s->d_maps) cudaFree(s->d_maps);
  if (s->d_flags) cudaFree(s->d_flags);
  if (s->d_timeline) cudaFree(s->d_timeline);
  if (s->host_ce) cudaFreeHost(s->host_ce);
  if (s->kv_fresh) cudaFree(s->kv_fresh);
  if (s->x_save) cudaFree(s->x_save);
  if (s->row_cos) cudaFree(s->row_cos);
  for (cudaEvent_t e : s->ev_pool) cudaEventDestroy(e);
  for (cudaEvent_t e : {s->ev_a, s->ev_b, s->ev_c, s->ev_d, s->ev_done[0], s->ev_done[1]})
    if (e) cudaEventDestroy(e);
  if (s->own_stream && s->st) cudaStreamDestroy(s->st);
  s->arena = nullptr;
  s->gemm_ws = nullptr;
  return DLLM_OK;
}

dllm_status upload_canvas(dllm_state* s) {
  std::vector<int32_t> canvas((size_t)s->b * s->T, s->m->cfg.vocab);
  for (int i = 0; i < s->b; ++i)
    std::memcpy(&canvas[(size_t)i * s->T], &s->prompts[(size_t)i * s->P], sizeof(int32_t) * s->P);
  CK(cudaMemcpyAsync(s->x, canvas.data(), canvas.size() * 4, cudaMemcpyHostToDevice, s->st));
  CK(cudaStreamSynchronize(s->st));
  return DLLM_OK;
}

void reset_counters(dllm_state* s) {
  s->remaining.assign((size_t)s->b * s->n_blocks, s->B);
}

dllm_status check_prompts(const dllm_model* m, const int32_t* prompts, int b, int P) {
  for (long long i = 0; i < (long long)b * P; ++i)
    if (prompts[i] < 0 || prompts[i] >= m->cfg.vocab) {
      set_error("prompt token %d at index %lld is outside [0, %d)", prompts[i], i, m->cfg.vocab);
      return DLLM_EINVAL;
    }
  return DLLM_OK;
}

}  // namespace

extern "C" dllm_status dllm_state_create(dllm_model* m, const int32_t* prompts, int32_t b, int32_t P,
                                         int32_t gen_len, int32_t block, void* stream, dllm_state** out) {
  if (!m || !out) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  *out = nullptr;
  if (b < 1 || P < 0 || gen_len < 0 || block < 1 || block > kMaxBlock || (gen_len > 0 && gen_len % block != 0) ||
      (long long)P + gen_len < 1 || (long long)P + gen_len > (1 << 20)) {
    set_error("bad shape: b=%d P=%d gen_len=%d block=%d (need b>=1, 1<=block<=%d, gen_len %% block == 0)", b, P,
              gen_len, block, kMaxBlock);
    return DLLM_EINVAL;
  }
  if (prompts) CKS(check_prompts(m, prompts, b, P));
  const dllm_config& c = m->cfg;
  dllm_state* s = new dllm_state();
  s->m = m;
  s->b = b;
  s->P = P;
  s->gen = gen_len;
  s->B = block;
  s->T = P + gen_len;
  s->n_blocks = gen_len / block;
  s->prompts.assign((size_t)b * P, 0);
  if (prompts) std::memcpy(s->prompts.data(), prompts, sizeof(int32_t) * b * P);
  reset_counters(s);

  const size_t d = c.d_model, F = m->F_pad, V = c.vocab, L = c.n_layers, H = c.n_heads, hd = c.head_dim;
  const size_t T = s->T, n_max = (size_t)b * T, n_lm = (size_t)b * block;
  const size_t v_tiles = (V + 127) / 128, d_tiles = d / 128;
  // fix-up counters: the largest tile grid of any GEMM of this state
  auto nt = [&](size_t n) { return (n + pick_bn((int)n, true) - 1) / pick_bn((int)n, true); };
  size_t cnt_n = std::max({(3 * d / 128) * nt(n_max), (2 * F / 128) * nt(n_max), (d / 128) * nt(n_max),
                           v_tiles * nt(n_lm)});
  // attention workspace: the largest plan among the row counts this state can use
  size_t attn_floats = 0, attn_cnt = 0;
  {
    std::vector<int> Rs = {block, (int)T};
    for (int j = 0; j < s->n_blocks; ++j) Rs.push_back((int)T - (P + j * block));
    for (int R : Rs) {
      if (R < 1) continue;
      AttnPlan a = plan_attention(b, (int)H, R, (int)T, m->sms);
      const size_t works = (size_t)b * H * a.q_tiles;
      attn_floats = std::max(attn_floats, works * a.splits * 16 * a.wq * (hd + 2));
      attn_cnt = std::max(attn_cnt, works);
    }
    // persistent step row sets: the block, two blocks (block-causal commit
    // forward + step)
    for (int R : {block, 2 * block}) {
      if (R < 1 || (long long)b * R > 128) continue;
      AttnPlan ap = plan_attention_persistent(b, (int)H, R, (int)T, m->sms);
      const size_t pworks = (size_t)b * H * ap.q_tiles;
      attn_floats = std::max(attn_floats, pworks * ap.splits * 16 * ap.wq * (hd + 2));
      attn_cnt = std::max(attn_cnt, pworks);
    }
    // row counts that take the tensor-core kernel
    for (int R : Rs) {
      if (R < kAttnTcMinRows) continue;
      AttnPlan at = plan_attention_tc(b, (int)H, R, (int)T, m->sms);
      if (at.splits < 2) continue;
      const size_t works = (size_t)tc_split_items(at, (long long)b * H * at.q_tiles);
      attn_floats = std::max(attn_floats, works * at.splits * 128 * (hd + 2));
      attn_cnt = std::max(attn_cnt, works);
    }
  }
  auto al = [](size_t bytes) { return (bytes + 1023) / 1024 * 1024; };
  size_t total = 0;
  const size_t o_x = total; total += al(n_max * 4);
  const size_t o_kv = total; total += al(L * 4 * b * H * T * hd * 2);
  const size_t o_h = total; total += al(n_max * d * 4);
  const size_t o_xn = total; total += al(2 * n_max * d * 2);
  const size_t o_ss = total; total += al(n_max * d_tiles * 4);
  const size_t o_q = total; total += al(2 * n_max * d * 2);
  const size_t o_ao = total; total += al(2 * n_max * d * 2);
  const size_t o_act = total; total += al(2 * n_max * F * 2);
  const size_t o_xf = total; total += al(2 * n_lm * d * 2);
  const size_t o_ssf = total; total += al(n_lm * d_tiles * 4);
  const size_t o_stm = total; total += al(v_tiles * n_lm * 4);
  const size_t o_sts = total; total += al(v_tiles * n_lm * 4);
  const size_t o_sta = total; total += al(v_tiles * n_lm * 4);
  const size_t o_conf = total; total += al(n_lm * 4);
  const size_t o_arg = total; total += al(n_lm * 4);
  const size_t o_ce = total; total += al((b + 1) * 4);
  const size_t o_sd = total; total += al(b * 4);
  const size_t o_gc = total; total += al(cnt_n * 4);
  const size_t o_ao2 = total; total += al(attn_floats * 4);
  const size_t o_ac = total; total += al(attn_cnt * 4);
  const size_t o_rope = total; total += al(T * (hd / 2) * 8);

  dllm_status st = dev_alloc(&s->arena, total);
  if (st != DLLM_OK) {
    delete s;
    return st;
  }
  st = dev_alloc((void**)&s->gemm_ws, (size_t)m->sms * 2 * 256 * 128 * 4);
  if (st != DLLM_OK) {
    state_free_device(s);
    delete s;
    return st;
  }
  uint8_t* a = static_cast<uint8_t*>(s->arena);
  s->x = reinterpret_cast<int32_t*>(a + o_x);
  s->kv = reinterpret_cast<uint16_t*>(a + o_kv);
  s->h = reinterpret_cast<float*>(a + o_h);
  s->xn = reinterpret_cast<uint16_t*>(a + o_xn);
  s->xn_lo = s->xn + n_max * d;
  s->ss = reinterpret_cast<float*>(a + o_ss);
  s->q = reinterpret_cast<uint16_t*>(a + o_q);
  s->q_lo = s->q + n_max * d;
  s->ao = reinterpret_cast<uint16_t*>(a + o_ao);
  s->ao_lo = s->ao + n_max * d;
  s->act = reinterpret_cast<uint16_t*>(a + o_act);
  s->act_lo = s->act + n_max * F;
  s->xf = reinterpret_cast<uint16_t*>(a + o_xf);
  s->xf_lo = s->xf + n_lm * d;
  s->ssf = reinterpret_cast<float*>(a + o_ssf);
  s->st_m = reinterpret_cast<float*>(a + o_stm);
  s->st_s = reinterpret_cast<float*>(a + o_sts);
  s->st_a = reinterpret_cast<int*>(a + o_sta);
  s->conf = reinterpret_cast<float*>(a + o_conf);
  s->arg = reinterpret_cast<int32_t*>(a + o_arg);
  s->count_err = reinterpret_cast<int32_t*>(a + o_ce);
  s->seq_done = reinterpret_cast<int*>(a + o_sd);
  s->gemm_cnt = reinterpret_cast<int*>(a + o_gc);
  s->attn_o = reinterpret_cast<float*>(a + o_ao2);
  s->attn_o_floats = attn_floats;
  s->attn_cnt_n = attn_cnt;
  s->attn_ml = s->attn_o;   // carved per launch from the same block (see run_attention)
  s->attn_cnt = reinterpret_cast<int*>(a + o_ac);
  s->rope = reinterpret_cast<float2*>(a + o_rope);

  auto fail = [&](dllm_status e) {
    state_free_device(s);
    delete s;
    return e;
  };
  if (stream) {
    s->st = static_cast<cudaStream_t>(stream);
  } else {
    if (cudaStreamCreateWithFlags(&s->st, cudaStreamNonBlocking) != cudaSuccess) {
      set_error("cudaStreamCreate failed");
      return fail(DLLM_ECUDA);
    }
    s->own_stream = true;
  }
  if (cudaMallocHost((void**)&s->host_ce, 2 * (b + 1) * 4) != cudaSuccess) {
    cudaGetLastError();
    set_error("cudaMallocHost failed");
    return fail(DLLM_ENOMEM);
  }
  if (cudaEventCreate(&s->ev_a) != cudaSuccess || cudaEventCreate(&s->ev_b) != cudaSuccess ||
      cudaEventCreate(&s->ev_c) != cudaSuccess || cudaEventCreate(&s->ev_d) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->ev_done[0], cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->ev_done[1], cudaEventDisableTiming) != cudaSuccess) {
    set_error("cudaEventCreate failed");
    return fail(DLLM_ECUDA);
  }
  if (cudaMemsetAsync(s->arena, 0, total, s->st) != cudaSuccess) {
    set_error("cudaMemset failed");
    return fail(DLLM_ECUDA);
  }
  // RoPE table: angle = pos * theta^(-2j/hd), rotate-half pairs (j, j + hd/2)
  {
    std::vector<float2> cs(T * (hd / 2));
    for (size_t pos = 0; pos < T; ++pos)
      for (size_t j = 0; j < hd / 2; ++j) {
        const double inv = std::pow((double)c.rope_theta, -2.0 * (double)j / (double)hd);
        const double ang = (double)pos * inv;
        cs[pos * (hd / 2) + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    if (cudaMemcpyAsync(s->rope, cs.data(), cs.size() * 8, cudaMemcpyHostToDevice, s->st) != cudaSuccess) {
      set_error("rope upload failed");
      return fail(DLLM_ECUDA);
    }
    if (cudaStreamSynchronize(s->st) != cudaSuccess) {
      set_error("stream sync failed");
      return fail(DLLM_ECUDA);
    }
  }
  if ((st = map_kv(&s->tm_kv, s->kv, hd, T, L * 4 * b * H, kStateAttnKT)) != DLLM_OK) return fail(st);
  if ((st = upload_canvas(s)) != DLLM_OK) return fail(st);
  *out = s;
  return DLLM_OK;
}

extern "C" void dllm_free_state(dllm_state* s) {
  if (!s) return;
  if (s->st) cudaStreamSynchronize(s->st);
  state_free_device(s);
  delete s;
}

extern "C" dllm_status dllm_state_reset(dllm_state* s, const int32_t* prompts) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  if (prompts) {
    CKS(check_prompts(s->m, prompts, s->b, s->P));
    std::memcpy(s->prompts.data(), prompts, sizeof(int32_t) * s->b * s->P);
  }
  reset_counters(s);
  CK(cudaMemsetAsync(s->kv, 0, (size_t)s->m->cfg.n_layers * 4 * s->b * s->m->cfg.d_model * s->T * 2, s->st));
  return upload_canvas(s);
}

namespace {

__global__ void set_prompts_kernel(int32_t* x, const int32_t* prompts, int b, int P, int T, int mask) {
  const long long n = (long long)b * T;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int seq = (int)(i / T), pos = (int)(i % T);
    x[i] = pos < P ? prompts[(long long)seq * P + pos] : mask;
  }
}

}  // namespace

extern "C" dllm_status dllm_state_set_prompts_device(dllm_state* s, const int32_t* prompts_dev) {
  if (!s || (!prompts_dev && s->P > 0)) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  reset_counters(s);
  const long long n = (long long)s->b * s->T;
  const int grid = (int)std::min<long long>((n + 255) / 256, 4096);
  set_prompts_kernel<<<grid, 256, 0, s->st>>>(s->x, prompts_dev, s->b, s->P, s->T, s->m->cfg.vocab);
  CK(cudaGetLastError());
  ++s->launches;
  return DLLM_OK;
}

// ====================================================================== pipeline
namespace {

cudaEvent_t next_event(dllm_state* s) {
  if (s->ev_next == s->ev_pool.size()) {
    cudaEvent_t e;
    cudaEventCreate(&e);
    s->ev_pool.push_back(e);
  }
  return s->ev_pool[s->ev_next++];
}

struct Timed {
  dllm_state* s;
  int cls;
  double bytes;
  cudaEvent_t e1 = nullptr;
  Timed(dllm_state* s_, int c, double b) : s(s_), cls(c), bytes(b) {
    if (s->timing) {
      cudaEvent_t e0 = next_event(s);
      e1 = next_event(s);
      cudaEventRecord(e0, s->st);
      s->pending.push_back({cls, {e0, e1}});
    }
  }
  ~Timed() {
    if (s->timing) cudaEventRecord(e1, s->st);
  }
};

void collect_timing(dllm_state* s) {
  for (size_t i = 0; i < s->pending.size(); ++i) {
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, s->pending[i].second.first, s->pending[i].second.second);
    const int c = s->pending[i].first;
    s->kt_ms[c] += ms;
    s->kt_n[c] += 1;
  }
  s->pending.clear();
  s->ev_next = 0;
}

const CUtensorMap* act_map(dllm_state* s, const void* base, int K, int N, int BN, dllm_status* st) {
  auto key = std::make_tuple(base, K, N, BN);
  auto it = s->act_maps.find(key);
  if (it != s->act_maps.end()) return &it->second;
  CUtensorMap m;
  *st = map_2d(&m, base, (uint64_t)K, (uint64_t)N, (uint32_t)BN);
  if (*st != DLLM_OK) return nullptr;
  return &(s->act_maps[key] = m);
}

// Same L1/shared split for the small kernels as for the GEMM and attention
// (a per-device function attribute: set once per device).
dllm_status pin_carveouts() {
  static std::mutex mu;
  static std::set<int> done;
  int dev = 0;
  CK(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(mu);
  if (done.count(dev)) return DLLM_OK;
  const void* ks[] = {(const void*)embed_kernel, (const void*)merge_select_kernel};
  for (const void* k : ks)
    CK(cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared));
  done.insert(dev);
  return DLLM_OK;
}

// Shape, work split and workspace fields of a GEMM's parameters.
void gemm_shape(dllm_state* s, GemmParams& p, int M, int K, int N, int BN) {
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = ceil_div(M, 128);
  p.n_tiles = ceil_div(N, BN);
  p.kc = ceil_div(K, 64);
  p.total = (long long)p.m_tiles * p.n_tiles * p.kc;
  p.ws = s->gemm_ws;
  p.counters = s->gemm_cnt;
  p.err = s->count_err + s->b;
  p.split = s->split ? 1 : 0;
}

dllm_status run_gemm(dllm_state* s, int kind, const CUtensorMap& tmA, int M, int K, const uint16_t* X,
                     const uint16_t* X_lo, int N, GemmParams p, int cls, double bytes) {
  const int BN = pick_bn(N, s->split);
  dllm_status st = DLLM_OK;
  const CUtensorMap* tmB = act_map(s, X, K, N, BN, &st);
  if (!tmB) return st;
  const CUtensorMap* tmBlo = tmB;
  if (s->split) {
    tmBlo = act_map(s, X_lo, K, N, BN, &st);
    if (!tmBlo) return st;
  }
  gemm_shape(s, p, M, K, N, BN);
  const int grid = (int)std::min<long long>(s->m->sms, p.total);
  if (p.total * (grid + 1) >= (1LL << 31)) {   // the kernel's stream-K arithmetic is 32-bit
    set_error("GEMM of %lld chunks is too large", (long long)p.total);
    return DLLM_EINVAL;
  }
  if (s->timing) s->kt_bytes[cls] += bytes;
  Timed t(s, cls, bytes);
  CK(launch_gemm(kind, BN, tmA, *tmB, *tmBlo, p, grid, s->st, true));
  ++s->launches;
  return DLLM_OK;
}


dllm_status run_attention(dllm_state* s, int layer, int R, int cls, double bytes) {
  const dllm_config& c = s->m->cfg;
  if (R >= kAttnTcMinRows) {
    const int d = c.d_model, n = s->b * R, bh = s->b * c.n_heads;
    dllm_status st = DLLM_OK;
    const CUtensorMap* tq = act_map(s, s->q, d, n, 128, &st);
    if (!tq) return st;
    const CUtensorMap* tqlo = tq;
    if (s->split) {
      tqlo = act_map(s, s->q_lo, d, n, 128, &st);
      if (!tqlo) return st;
    }
    auto it = s->kv64_maps.find(s->kv);
    if (it == s->kv64_maps.end()) {
      CUtensorMap m;
      CKS(map_kv(&m, s->kv, c.head_dim, s->T, (uint64_t)c.n_layers * 4 * bh, 64));
      it = s->kv64_maps.emplace(s->kv, m).first;
    }
    AttnPlan at = plan_attention_tc(s->b, c.n_heads, R, s->T, s->m->sms);
    const long long tc_items = (long long)s->b * c.n_heads * at.q_tiles;
    const size_t tc_works = (size_t)tc_split_items(at, tc_items);
    if (at.splits > 1 &&
        (tc_works * at.splits * 128 * (c.head_dim + 2) > s->attn_o_floats || tc_works > s->attn_cnt_n)) {
      set_error("attention merge workspace too small for %d rows", R);
      return DLLM_EINVAL;
    }
    AttnParams p = {};
    p.q = s->q;
    p.q_lo = s->split ? s->q_lo : nullptr;
    p.kv_lo = s->split ? 1 : 0;
    p.o = s->ao;
    p.o_lo = s->split ? s->ao_lo : nullptr;
    p.R = R;
    p.b = s->b;
    p.H = c.n_heads;
    p.T = s->T;
    p.q_tiles = at.q_tiles;
    p.splits = at.splits;
    p.kps = at.kps;
    p.n_whole = (int)at.n_whole;
    p.ws_o = s->attn_o;
    p.ws_ml = s->attn_o + (long long)tc_works * at.splits * 128 * c.head_dim;
    p.counters = s->attn_cnt;
    p.z_k0 = ((layer * 2 + 0) * 2 + 0) * bh;
    p.z_kl0 = ((layer * 2 + 0) * 2 + 1) * bh;
    p.z_v0 = ((layer * 2 + 1) * 2 + 0) * bh;
    p.z_vl0 = ((layer * 2 + 1) * 2 + 1) * bh;
    p.row0 = s->last_row0;
    p.mask_P = s->P;
    p.mask_B = s->block_causal ? s->B : 0;
    p.scale_log2 = kLog2e / std::sqrt((float)c.head_dim);
    p.err = s->count_err + s->b;
    if (s->timing) s->kt_bytes[cls] += bytes;
    Timed t(s, cls, bytes);
    CK(launch_attention_tc(c.head_dim, *tq, *tqlo, it->second, it->second, p, dim3((unsigned)tc_ctas(at, tc_items)),
                           s->st, true));
    ++s->launches;
    return DLLM_OK;
  }
  AttnPlan a = plan_attention(s->b, c.n_heads, R, s->T, s->m->sms);
  const int QT = 16 * a.wq;
  const long long works = (long long)s->b * c.n_heads * a.q_tiles;
  AttnParams p = {};
  p.q = s->q;
  p.q_lo = s->split ? s->q_lo : nullptr;
  p.kv_lo = s->split ? 1 : 0;
  p.o = s->ao;
  p.o_lo = s->split ? s->ao_lo : nullptr;
  p.R = R;
  p.b = s->b;
  p.H = c.n_heads;
  p.T = s->T;
  const int bh = s->b * c.n_heads;
  p.z_k0 = ((layer * 2 + 0) * 2 + 0) * bh;
  p.z_kl0 = ((layer * 2 + 0) * 2 + 1) * bh;
  p.z_v0 = ((layer * 2 + 1) * 2 + 0) * bh;
  p.z_vl0 = ((layer * 2 + 1) * 2 + 1) * bh;
  p.q_tiles = a.q_tiles;
  p.splits = a.splits;
  p.kps = a.kps;
  p.row0 = s->last_row0;
  p.mask_P = s->P;
  p.mask_B = s->block_causal ? s->B : 0;
  p.scale_log2 = kLog2e / std::sqrt((float)c.head_dim);
  p.ws_o = s->attn_o;
  p.ws_ml = s->attn_o + works * a.splits * QT * c.head_dim;
  p.counters = s->attn_cnt;
  p.err = s->count_err + s->b;
  if (s->timing) s->kt_bytes[cls] += bytes;
  Timed t(s, cls, bytes);
  CK(launch_attention(c.head_dim, a.wq, kStateAttnKT, s->tm_kv, s->tm_kv, p,
                      dim3(a.splits, a.q_tiles * c.n_heads, s->b), s->st, true));
  ++s->launches;
  return DLLM_OK;
}

// Forward over rows [row0, row0 + R) of every sequence.  refresh: write K/V
// only (stop after the last layer's QKV).  Otherwise finish with the LM head
// on the block rows [blk, blk + B) and select/commit with `rule`.
dllm_status run_forward(dllm_state* s, int row0, int R, bool refresh, int blk, const SelectRule& rule) {
  const dllm_model* m = s->m;
  const dllm_config& c = m->cfg;
  const int d = c.d_model, L = c.n_layers, F = m->F_pad, V = c.vocab;
  const int n = s->b * R, n_lm = s->b * s->B;
  const double wb = 2.0;  // bf16
  const int co = (refresh || s->fused_fwd) ? KC_REFRESH : 0;
  CKS(pin_carveouts());
  s->last_row0 = row0;
  s->last_R = R;
  s->last_blk = blk;
  {
    EmbedParams e{s->x, m->embed, m->layers[0].attn_norm, s->h, s->xn, s->split ? s->xn_lo : nullptr, s->ss,
                  d, R, row0, s->T};
    Timed t(s, co + KC_EMBED, (double)n * d * (2 + 4 + 2));
    if (s->timing) s->kt_bytes[co + KC_EMBED] += (double)n * d * 8;
    CK(launch_ex(embed_kernel, dim3(n), dim3(d / 8), 0, s->st, true, e));
    ++s->launches;
  }
  if (s->trace) CK(cudaMemcpyAsync(s->trace_buf, s->h, (size_t)n * d * 4, cudaMemcpyDeviceToDevice, s->st));
  // algorithmic K/V bytes: K and V once, bf16 (the split's low halves are an
  // implementation cost, not counted)
  const double kv_bytes = (double)s->b * s->T * d * 2 * 2;
  for (int l = 0; l < L; ++l) {
    const LayerW& w = m->layers[l];
    const bool last = l == L - 1;
    GemmParams p = {};
    p.ss_in = s->ss;
    p.ss_in_tiles = d / 128;
    p.inv_d = 1.0f / d;
    p.eps = c.norm_eps;
    p.R = R;
    p.row0 = row0;
    p.q_out = s->q;
    p.q_out_lo = s->split ? s->q_lo : nullptr;
    p.kv = s->kv;
    p.rope_cs = s->rope;
    p.d_model = d;
    p.head_dim = c.head_dim;
    p.n_heads = c.n_heads;
    p.T_pad = s->T;
    p.b_seqs = s->b;
    p.layer = l;
    CKS(run_gemm(s, GEMM_QKV, w.tm_qkv, 3 * d, d, s->xn, s->xn_lo, n, p, co + KC_QKV,
                 3.0 * d * d * wb + (double)n * d * wb * 4));
    if (refresh && last) break;
    CKS(run_attention(s, l, R, co + KC_ATTN, kv_bytes + (double)n * d * wb * 2));
    GemmParams o = {};
    o.R = R;
    o.row0 = row0;
    o.d_model = d;
    o.h = s->h;
    o.g_next = w.ffn_norm;
    o.xn_out = s->xn;
    o.xn_out_lo = s->split ? s->xn_lo : nullptr;
    o.ss_out = s->ss;
    CKS(run_gemm(s, GEMM_RESID, w.tm_o, d, d, s->ao, s->ao_lo, n, o, co + KC_O,
                 (double)d * d * wb + (double)n * d * (wb + 8 + wb)));
    GemmParams gu = {};
    gu.ss_in = s->ss;
    gu.ss_in_tiles = d / 128;
    gu.inv_d = 1.0f / d;
    gu.eps = c.norm_eps;
    gu.act = s->act;
    gu.act_lo = s->split ? s->act_lo : nullptr;
    gu.act_ld = F;
    CKS(run_gemm(s, GEMM_SWIGLU, w.tm_gu, 2 * F, d, s->xn, s->xn_lo, n, gu, co + KC_GU,
                 2.0 * F * d * wb + (double)n * (d + F) * wb));
    GemmParams dn = {};
    dn.R = R;
    dn.row0 = row0;
    dn.d_model = d;
    dn.h = s->h;
    if (last) {
      dn.g_next = m->final_norm;
      dn.xn_out = s->xf;
      dn.xn_out_lo = s->split ? s->xf_lo : nullptr;
      dn.ss_out = s->ssf;
      dn.remap = 1;
      dn.blk_start = blk;
      dn.blk_len = s->B;
    } else {
      dn.g_next = m->layers[l + 1].attn_norm;
      dn.xn_out = s->xn;
      dn.xn_out_lo = s->split ? s->xn_lo : nullptr;
      dn.ss_out = s->ss;
    }
    CKS(run_gemm(s, GEMM_RESID, w.tm_d, d, F, s->act, s->act_lo, n, dn, co + KC_D,
                 (double)d * F * wb + (double)n * (F * wb + 8.0 * d + wb * d)));
    if (s->trace)
      CK(cudaMemcpyAsync(s->trace_buf + (size_t)(l + 1) * n * d, s->h, (size_t)n * d * 4, cudaMemcpyDeviceToDevice,
                         s->st));
  }
  if (refresh) return DLLM_OK;
  GemmParams lm = {};
  lm.ss_in = s->ssf;
  lm.ss_in_tiles = d / 128;
  lm.inv_d = 1.0f / d;
  lm.eps = c.norm_eps;
  lm.st_m = s->st_m;
  lm.st_s = s->st_s;
  lm.st_a = s->st_a;
  CKS(run_gemm(s, GEMM_LMHEAD, m->tm_lm, V, d, s->xf, s->xf_lo, n_lm, lm, KC_LM, (double)V * d * wb + (double)n_lm * d * wb));
  MergeParams mp = {};
  mp.st_m = s->st_m;
  mp.st_s = s->st_s;
  mp.st_a = s->st_a;
  mp.v_tiles = ceil_div(V, 128);
  mp.n_rows = n_lm;
  mp.B = s->B;
  mp.T = s->T;
  mp.blk_start = blk;
  mp.mask_id = V;
  mp.x = s->x;
  mp.conf = s->conf;
  mp.arg = s->arg;
  mp.count = s->count_err;
  mp.seq_done = s->seq_done;
  mp.rule = rule;
  {
    Timed t(s, KC_MERGE, (double)mp.v_tiles * n_lm * 12);
    if (s->timing) s->kt_bytes[KC_MERGE] += (double)mp.v_tiles * n_lm * 12;
    CK(launch_ex(merge_select_kernel, dim3(n_lm), dim3(256), 0, s->st, true, mp));
    ++s->launches;
  }
  return DLLM_OK;
}

// Rows of the persistent step of kind k for block j: (first row position,
// rows per sequence); rows = 0 when that step does not run persistent.
//   SK_DUAL    the block's B rows (DualCache);
//   SK_COMMIT  block j-1 and block j (2B rows) under the block-causal mask:
//              block j-1's commit forward fused with block j's first step.
// (PrefixCache steps over rows [block start, T) were measured on this kernel
// too, for up to 128 and up to 64 rows: no faster than the per-kernel path.)
std::pair<int, int> step_rows(const dllm_state* s, int k, int j) {
  const int blk = s->P + j * s->B;
  int row0 = blk, R = s->B;
  if (k == SK_COMMIT) {
    if (j == 0) return {0, 0};
    row0 = blk - s->B;
    R = 2 * s->B;
  }
  // at most 128 activation rows per tile; the fused merge and select handle
  // blocks of up to 32 positions
  if ((long long)s->b * R > 128 || s->B > 32) return {0, 0};
  return {row0, R};
}

// Tensor-map table and per-kind, per-block phase lists of the persistent step.
dllm_status build_step(dllm_state* s) {
  const dllm_model* m = s->m;
  const dllm_config& c = m->cfg;
  const int d = c.d_model, L = c.n_layers, F = m->F_pad, V = c.vocab;
  const int n_lm = s->b * s->B;
  std::vector<CUtensorMap> maps;
  auto add = [&](const CUtensorMap& t) {
    maps.push_back(t);
    return (int)maps.size() - 1;
  };
  std::vector<int> i_qkv(L), i_o(L), i_gu(L), i_d(L);
  for (int l = 0; l < L; ++l) {
    i_qkv[l] = add(m->layers[l].tm_qkv);
    i_o[l] = add(m->layers[l].tm_o);
    i_gu[l] = add(m->layers[l].tm_gu);
    i_d[l] = add(m->layers[l].tm_d);
  }
  const int i_lm = add(m->tm_lm);
  s->map_kv = add(s->tm_kv);
  CUtensorMap t;
  // activation maps per (rows, tile rows): xn, xn_lo, ao, ao_lo, act, act_lo over n rows; xf, xf_lo over the block rows
  std::map<std::pair<int, int>, std::array<int, 8>> act_maps;
  auto act_for = [&](int n, int BN, std::array<int, 8>* out) -> dllm_status {
    auto it = act_maps.find({n, BN});
    if (it != act_maps.end()) {
      *out = it->second;
      return DLLM_OK;
    }
    std::array<int, 8> ix;
    const uint16_t* base[8] = {s->xn, s->xn_lo, s->ao, s->ao_lo, s->act, s->act_lo, s->xf, s->xf_lo};
    const int K[8] = {d, d, d, d, F, F, d, d};
    for (int i = 0; i < 8; ++i) {
      CKS(map_2d(&t, base[i], K[i], i < 6 ? n : n_lm, BN));
      ix[i] = add(t);
    }
    act_maps.emplace(std::make_pair(n, BN), ix);
    *out = ix;
    return DLLM_OK;
  };

  const int n_phases = 5 * L + 3;
  const int NB = s->n_blocks;
  std::vector<StepPhase> ph((size_t)SK_KINDS * NB * n_phases);
  std::vector<StepShape> shapes((size_t)SK_KINDS * NB);
  for (int kind = 0; kind < SK_KINDS; ++kind)
  for (int j = 0; j < NB; ++j) {
    const auto rr = step_rows(s, kind, j);
    if (rr.second == 0) continue;
    const int blk = s->P + j * s->B;      // the block whose step this is (LM head, select)
    const int row0 = rr.first, R = rr.second;
    const int n = s->b * R;
    const int BN = pick_bn(n, true);
    std::array<int, 8> ix;
    CKS(act_for(n, BN, &ix));
    const int i_xn = ix[0], i_xnl = ix[1], i_ao = ix[2], i_aol = ix[3], i_act = ix[4], i_actl = ix[5], i_xf = ix[6],
              i_xfl = ix[7];
    StepShape& sh = shapes[(size_t)kind * NB + j];
    sh.bn = BN;
    sh.rows = R;
    sh.row0 = row0;
    sh.ap = plan_attention_persistent(s->b, c.n_heads, R, s->T, s->m->sms);
    StepPhase* P = &ph[((size_t)kind * NB + j) * n_phases];
    int k = 0;
    P[k] = StepPhase{};
    P[k++].kind = PH_EMBED;
    for (int l = 0; l < L; ++l) {
      const LayerW& w = m->layers[l];
      const bool last = l == L - 1;
      StepPhase q = {};
      q.kind = PH_GEMM;
      q.gemm_kind = GEMM_QKV;
      q.map_a = i_qkv[l];
      q.map_b = i_xn;
      q.map_blo = i_xnl;
      gemm_shape(s, q.g, 3 * d, d, n, BN);
      q.g.ss_in = s->ss;
      q.g.ss_in_tiles = d / 128;
      q.g.inv_d = 1.0f / d;
      q.g.eps = c.norm_eps;
      q.g.R = R;
      q.g.row0 = row0;
      q.g.q_out = s->q;
      q.g.q_out_lo = s->split ? s->q_lo : nullptr;
      q.g.kv = s->kv;
      q.g.rope_cs = s->rope;
      q.g.d_model = d;
      q.g.head_dim = c.head_dim;
      q.g.n_heads = c.n_heads;
      q.g.T_pad = s->T;
      q.g.b_seqs = s->b;
      q.g.layer = l;
      P[k++] = q;
      StepPhase at = {};
      at.kind = PH_ATTN;
      at.layer = l;
      P[k++] = at;
      StepPhase o = {};
      o.kind = PH_GEMM;
      o.gemm_kind = GEMM_RESID;
      o.map_a = i_o[l];
      o.map_b = i_ao;
      o.map_blo = i_aol;
      gemm_shape(s, o.g, d, d, n, BN);
      o.g.R = R;
      o.g.row0 = row0;
      o.g.d_model = d;
      o.g.h = s->h;
      o.g.g_next = w.ffn_norm;
      o.g.xn_out = s->xn;
      o.g.xn_out_lo = s->split ? s->xn_lo : nullptr;
      o.g.ss_out = s->ss;
      P[k++] = o;
      StepPhase gu = {};
      gu.kind = PH_GEMM;
      gu.gemm_kind = GEMM_SWIGLU;
      gu.map_a = i_gu[l];
      gu.map_b = i_xn;
      gu.map_blo = i_xnl;
      gemm_shape(s, gu.g, 2 * F, d, n, BN);
      gu.g.ss_in = s->ss;
      gu.g.ss_in_tiles = d / 128;
      gu.g.inv_d = 1.0f / d;
      gu.g.eps = c.norm_eps;
      gu.g.act = s->act;
      gu.g.act_lo = s->split ? s->act_lo : nullptr;
      gu.g.act_ld = F;
      P[k++] = gu;
      StepPhase dn = {};
      dn.kind = PH_GEMM;
      dn.gemm_kind = GEMM_RESID;
      dn.map_a = i_d[l];
      dn.map_b = i_act;
      dn.map_blo = i_actl;
      gemm_shape(s, dn.g, d, F, n, BN);
      dn.g.R = R;
      dn.g.row0 = row0;
      dn.g.d_model = d;
      dn.g.h = s->h;
      if (last) {
        dn.g.g_next = m->final_norm;
        dn.g.xn_out = s->xf;
        dn.g.xn_out_lo = s->split ? s->xf_lo : nullptr;
        dn.g.ss_out = s->ssf;
        dn.g.remap = 1;
        dn.g.blk_start = blk;
        dn.g.blk_len = s->B;
      } else {
        dn.g.g_next = m->layers[l + 1].attn_norm;
        dn.g.xn_out = s->xn;
        dn.g.xn_out_lo = s->split ? s->xn_lo : nullptr;
        dn.g.ss_out = s->ss;
      }
      P[k++] = dn;
    }
    StepPhase lm = {};
    lm.kind = PH_GEMM;
    lm.gemm_kind = GEMM_LMHEAD;
    lm.map_a = i_lm;
    lm.map_b = i_xf;
    lm.map_blo = i_xfl;
    gemm_shape(s, lm.g, V, d, n_lm, BN);
    lm.g.ss_in = s->ssf;
    lm.g.ss_in_tiles = d / 128;
    lm.g.inv_d = 1.0f / d;
    lm.g.eps = c.norm_eps;
    lm.g.st_m = s->st_m;
    lm.g.st_s = s->st_s;
    lm.g.st_a = s->st_a;
    P[k++] = lm;
    P[k] = StepPhase{};
    P[k++].kind = PH_MERGE;
  }
  // Dataflow flags (one int block, zeroed per launch; the same layout for
  // every block's phase list, whose order is embed, L x [QKV, ATTN, O, GU, D],
  // LM, MERGE).  A GEMM phase owns m_tiles row-tile flags (each counts its
  // finished n-tiles), a completion counter and m_tiles * n_tiles stream-K
  // fix-up counters; an attention phase owns one flag per head (counting
  // finished works) and a completion counter; the embedding one counter (one
  // count per CTA).
  const int G = s->m->sms;
  std::vector<int> cnt_of(n_phases, -1), unit_of(n_phases, -1), done_of(n_phases, -1);
  int n_flags = 0;
  size_t first = 0;
  while (first < shapes.size() && shapes[first].rows == 0) ++first;
  if (first == shapes.size()) {
    set_error("persistent step: no block fits");
    return DLLM_EINVAL;
  }
  for (int k = 0; k < n_phases; ++k) {
    const StepPhase& q = ph[first * n_phases + k];
    if (q.kind == PH_GEMM && q.g.n_tiles != 1) {
      set_error("persistent step: %d activation tiles in a phase", q.g.n_tiles);
      return DLLM_EINVAL;
    }
    if (q.kind == PH_EMBED) {
      done_of[k] = n_flags++;
    } else if (q.kind == PH_ATTN) {
      unit_of[k] = n_flags;
      n_flags += c.n_heads;
      done_of[k] = n_flags++;
    } else if (q.kind == PH_GEMM) {
      if (q.g.total * (G + 1) >= (1LL << 31)) {   // the kernel's stream-K arithmetic is 32-bit
        set_error("persistent step: %lld chunks in one phase is too many", (long long)q.g.total);
        return DLLM_EINVAL;
      }
      unit_of[k] = n_flags;
      n_flags += q.g.m_tiles;
      done_of[k] = n_flags++;
      cnt_of[k] = n_flags;
      n_flags += q.g.m_tiles * q.g.n_tiles;
    }
  }
  if (s->n_flags < n_flags) {
    if (s->d_flags) cudaFree(s->d_flags);
    s->d_flags = nullptr;
    s->n_flags = 0;
    CKS(dev_alloc((void**)&s->d_flags, (size_t)n_flags * 4));
    s->n_flags = n_flags;
  }
  for (size_t li = 0; li < shapes.size(); ++li) {
    if (shapes[li].rows == 0) continue;
    const int BN = shapes[li].bn;
    const AttnPlan& ap = shapes[li].ap;
    StepPhase* P = &ph[li * n_phases];
    int gemm_ord = 0;
    for (int k = 0; k < n_phases; ++k) {
      StepPhase& q = P[k];
      q.unit0 = unit_of[k];
      q.done = done_of[k];
      q.rs_done = -1;
      q.rs_need = 0;
      q.dep0 = 0;
      q.dep_shift = 31;
      q.dep_need = 0;
      q.dep_attn = 0;
      q.qkv0 = 0;
      q.qkv_need = 0;
      q.src_done = 0;
      q.src_need = 0;
      if (q.kind == PH_MERGE) {           // every LM-head tile
        const StepPhase& lm = P[k - 1];
        q.rs_done = done_of[k - 1];
        q.rs_need = lm.g.m_tiles * lm.g.n_tiles;
        continue;
      }
      if (q.kind == PH_ATTN) {            // q, k, v row tiles of the QKV phase before
        q.qkv0 = unit_of[k - 1];
        q.qkv_need = P[k - 1].g.n_tiles;
        continue;
      }
      if (q.kind != PH_GEMM) continue;
      GemmParams& g = q.g;
      g.counters = s->d_flags + cnt_of[k];
      g.ws = s->gemm_ws + (size_t)(gemm_ord++ & 1) * G * 2 * BN * 128;
      const StepPhase& prev = P[k - 1];
      q.src_done = done_of[k - 1];
      q.src_need = prev.kind == PH_EMBED  ? G
                   : prev.kind == PH_ATTN ? s->b * ap.q_tiles * c.n_heads   // attention works (seq, head, query tile)
                                          : prev.g.m_tiles * prev.g.n_tiles;
      if (prev.kind == PH_EMBED) {        // QKV of layer 0: every CTA's embedding rows
        q.dep0 = done_of[k - 1];
        q.dep_shift = 31;                 // every chunk: unit 0, the embedding counter
        q.dep_need = G;
        q.rs_done = done_of[k - 1];
        q.rs_need = G;
      } else if (prev.kind == PH_ATTN) {  // O: this layer's attention heads
        q.dep0 = unit_of[k - 1];
        q.dep_shift = c.head_dim == 128 ? 1 : 0;   // a head spans head_dim columns
        q.dep_need = s->b * ap.q_tiles;
        q.dep_attn = 1;
        q.layer = prev.layer;
      } else {                            // QKV (l > 0), GU, D, LM: the GEMM before
        q.dep0 = unit_of[k - 1];
        q.dep_shift = prev.gemm_kind == GEMM_SWIGLU ? 0 : 1;   // a SwiGLU tile writes 64 columns, others 128
        q.dep_need = prev.g.n_tiles;
        if (g.ss_in) {                    // row factors from every tile of the RESID phase before
          q.rs_done = done_of[k - 1];
          q.rs_need = prev.g.m_tiles * prev.g.n_tiles;
        }
      }
    }
  }
  if (s->d_phases) cudaFree(s->d_phases);
  if (s->d_maps) cudaFree(s->d_maps);
  s->d_phases = nullptr;
  s->d_maps = nullptr;
  CKS(dev_alloc((void**)&s->d_phases, ph.size() * sizeof(StepPhase)));
  CKS(dev_alloc((void**)&s->d_maps, maps.size() * sizeof(CUtensorMap)));
  CK(cudaMemcpy(s->d_phases, ph.data(), ph.size() * sizeof(StepPhase), cudaMemcpyHostToDevice));
  CK(cudaMemcpy(s->d_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice));
  s->n_phases = n_phases;
  s->step_shape = shapes;
  s->step_split = s->split;
  s->step_built = true;
  return DLLM_OK;
}

// The persistent step of kind k runs block j's step when its rows fit.
bool use_persistent(const dllm_state* s, int kind, int j) {
  return s->persistent && !s->trace && step_rows(s, kind, j).second > 0;
}

// One denoise step of block j as a single cooperative launch: DualCache, or
// (block-causal) block j-1's commit forward with block j's first step.
dllm_status run_step_persistent(dllm_state* s, int j, const SelectRule& rule, int kind, bool skip_done = false) {
  if (!s->step_built || s->step_split != s->split) CKS(build_step(s));
  const dllm_model* m = s->m;
  const dllm_config& c = m->cfg;
  const int d = c.d_model, V = c.vocab;
  const int blk = s->P + j * s->B;
  const int n = s->b * s->B;
  const size_t li = (size_t)kind * s->n_blocks + j;
  const StepShape& sh = s->step_shape[li];
  if (sh.rows == 0) {
    set_error("no persistent step of kind %d for block %d", kind, j);
    return DLLM_EINVAL;
  }
  s->last_row0 = sh.row0;
  s->last_R = sh.rows;
  s->last_blk = blk;
  StepArgs a = {};
  a.phases = s->d_phases + li * s->n_phases;
  a.n_phases = s->n_phases;
  a.maps = s->d_maps;
  a.flags = s->d_flags;
  a.err = s->count_err + s->b;
  a.emb = EmbedParams{s->x, m->embed, m->layers[0].attn_norm, s->h, s->xn, s->split ? s->xn_lo : nullptr, s->ss,
                      d, sh.rows, sh.row0, s->T};
  const AttnPlan& ap = sh.ap;
  const int QT = 32;
  const long long works = (long long)s->b * c.n_heads * ap.q_tiles;
  a.attn.q = s->q;
  a.attn.q_lo = s->split ? s->q_lo : nullptr;
  a.attn.kv_lo = s->split ? 1 : 0;
  a.attn.o = s->ao;
  a.attn.o_lo = s->split ? s->ao_lo : nullptr;
  a.attn.R = sh.rows;
  a.attn.b = s->b;
  a.attn.H = c.n_heads;
  a.attn.T = s->T;
  a.attn.row0 = sh.row0;
  a.attn.mask_P = s->P;
  a.attn.mask_B = s->block_causal ? s->B : 0;
  a.attn.q_tiles = ap.q_tiles;
  a.attn.splits = ap.splits;
  a.attn.kps = ap.kps;
  a.attn.scale_log2 = kLog2e / std::sqrt((float)c.head_dim);
  a.attn.ws_o = s->attn_o;
  a.attn.ws_ml = s->attn_o + works * ap.splits * QT * c.head_dim;
  a.attn.counters = s->attn_cnt;
  a.attn.err = s->count_err + s->b;
  a.attn_map = s->map_kv;
  a.attn_items = (int)(works * ap.splits);
  a.merge.st_m = s->st_m;
  a.merge.st_s = s->st_s;
  a.merge.st_a = s->st_a;
  a.merge.v_tiles = ceil_div(V, 128);
  a.merge.n_rows = n;
  a.merge.B = s->B;
  a.merge.T = s->T;
  a.merge.blk_start = blk;
  a.merge.mask_id = V;
  a.merge.x = s->x;
  a.merge.conf = s->conf;
  a.merge.arg = s->arg;
  a.merge.count = s->count_err;
  a.merge.seq_done = s->seq_done;
  a.merge.rule = rule;
  a.prefetch = s->step_prefetch;
  a.skip_done = skip_done ? 1 : 0;
  if (s->timeline) {
    const size_t tl_bytes = (size_t)s->m->sms * s->n_phases * kTimelineSlots * 8;
    if (!s->d_timeline) CKS(dev_alloc((void**)&s->d_timeline, tl_bytes));
    CK(cudaMemsetAsync(s->d_timeline, 0, tl_bytes, s->st));
    a.timeline = s->d_timeline;
  }
  CK(cudaMemsetAsync(s->d_flags, 0, (size_t)s->n_flags * 4, s->st));
  const double bytes = (double)s->m->cfg.n_layers * 2.0 *
                           (4.0 * d * d + 3.0 * (double)d * c.d_ffn) +
                       2.0 * V * d + (double)s->b * s->T * d * 2 * 2 * c.n_layers;   // K/V once, bf16
  if (s->timing) s->kt_bytes[KC_PSTEP] += bytes;
  Timed t(s, KC_PSTEP, bytes);
  const int grid = s->m->sms;
  cudaError_t e = c.head_dim == 64 ? launch_step_hd64(sh.bn, a, grid, s->st)
                                   : launch_step_hd128(sh.bn, a, grid, s->st);
  CK(e);
  ++s->launches;
  return DLLM_OK;
}

dllm_status finish_sync(dllm_state* s) {
  CK(cudaMemcpyAsync(s->host_ce, s->count_err, (s->b + 1) * 4, cudaMemcpyDeviceToHost, s->st));
  CK(cudaStreamSynchronize(s->st));
  if (s->timing) collect_timing(s);
  if (s->host_ce[s->b] != 0) {
    set_error("a kernel gave up a bounded wait (site %d); outputs are invalid", s->host_ce[s->b]);
    return DLLM_ETIMEOUT;
  }
  return DLLM_OK;
}

dllm_status to_rule(const dllm_select* sel, SelectRule* r) {
  if (!sel) {
    set_error("selection rule is NULL");
    return DLLM_EINVAL;
  }
  r->policy = sel->policy;
  r->tau = sel->tau;
  r->k = sel->k;
  r->factor = sel->factor;
  if (sel->policy < 0 || sel->policy > 4 || (sel->policy == 0 && std::isnan(sel->tau)) ||
      ((sel->policy == 1 || sel->policy == 4) && sel->k < 1) || (sel->policy == 2 && !(sel->factor > 0))) {
    set_error("bad selection rule: policy=%d tau=%f k=%d factor=%f", sel->policy, sel->tau, sel->k, sel->factor);
    return DLLM_EINVAL;
  }
  return DLLM_OK;
}

dllm_status do_refresh(dllm_state* s, cudaEvent_t e0 = nullptr, cudaEvent_t e1 = nullptr) {
  if (s->T < 1) return DLLM_OK;
  SelectRule none{0, 2.0f, 1, 1.0f};
  if (e0) CK(cudaEventRecord(e0, s->st));
  CK(cudaMemsetAsync(s->count_err + s->b, 0, 4, s->st));
  CKS(run_forward(s, 0, s->T, true, 0, none));
  if (e1) CK(cudaEventRecord(e1, s->st));
  return finish_sync(s);
}

// commit_prev (block-causal runs, dllm_run): block j-1's commit forward runs
// in the same persistent launch as this step (the caller checked it fits).
// Enqueue one denoise step of block j on the state's stream without waiting
// for it: its counts and error word are copied to host slot `slot`, and
// ev_done[slot] is recorded after them.  skip_done: the step is launched
// before the previous step's counts were read (a persistent DualCache step
// only); it does nothing when block j no longer holds a MASK.
dllm_status step_enqueue(dllm_state* s, int j, const SelectRule& rule, int mode, bool commit_prev, bool skip_done,
                         int slot, cudaEvent_t e0, cudaEvent_t e1) {
  if (j < 0 || j >= s->n_blocks) {
    set_error("block_idx %d outside [0, %d)", j, s->n_blocks);
    return DLLM_EINVAL;
  }
  if (mode < 0 || mode > 2) {
    set_error("bad cache mode %d", mode);
    return DLLM_EINVAL;
  }
  const int blk = s->P + j * s->B;
  int row0, R;
  if (mode == DLLM_CACHE_DUAL) {
    row0 = blk;
    R = s->B;
  } else if (mode == DLLM_CACHE_PREFIX) {
    row0 = blk;
    R = s->T - blk;
  } else {
    row0 = 0;
    R = s->T;
  }
  const int kind = commit_prev ? SK_COMMIT : mode == DLLM_CACHE_DUAL ? SK_DUAL : -1;
  if (commit_prev && !use_persistent(s, SK_COMMIT, j)) {
    set_error("block %d: the fused commit forward does not fit one launch", j);
    return DLLM_EINVAL;
  }
  const bool persistent = kind >= 0 && use_persistent(s, kind, j);
  if (skip_done && (kind != SK_DUAL || !persistent)) {
    set_error("block %d: only a persistent DualCache step can be launched ahead", j);
    return DLLM_EINVAL;
  }
  if (e0) CK(cudaEventRecord(e0, s->st));
  CK(cudaMemsetAsync(s->count_err, 0, (s->b + 1) * 4, s->st));
  if (persistent) {
    CKS(run_step_persistent(s, j, rule, kind, skip_done));
  } else {
    CKS(run_forward(s, row0, R, false, blk, rule));
  }
  if (e1) CK(cudaEventRecord(e1, s->st));
  CK(cudaMemcpyAsync(s->host_ce + (size_t)slot * (s->b + 1), s->count_err, (s->b + 1) * 4, cudaMemcpyDeviceToHost,
                     s->st));
  CK(cudaEventRecord(s->ev_done[slot], s->st));
  return DLLM_OK;
}

// Wait for the step whose counts go to host slot `slot` and apply them to
// block j's MASK counts.
dllm_status step_collect(dllm_state* s, int j, const SelectRule& rule, int slot, int32_t* committed, int* total) {
  CK(cudaEventSynchronize(s->ev_done[slot]));
  if (s->timing) collect_timing(s);
  const int32_t* ce = s->host_ce + (size_t)slot * (s->b + 1);
  if (ce[s->b] != 0) {
    set_error("a kernel gave up a bounded wait (site %d); outputs are invalid", ce[s->b]);
    return DLLM_ETIMEOUT;
  }
  int sum = 0;
  for (int i = 0; i < s->b; ++i) {
    const int cnt = ce[i];
    int& rem = s->remaining[(size_t)i * s->n_blocks + j];
    // every rule commits at least one MASK of the block per step, except the
    // scheduled one, which may commit none while more steps are left
    if (cnt > rem || (rem > 0 && cnt == 0 && !(rule.policy == 4 && rule.k > 1))) {
      set_error("sequence %d committed %d with %d MASK left in block %d", i, cnt, rem, j);
      return DLLM_ESTATE;
    }
    rem -= cnt;
    sum += cnt;
    if (committed) committed[i] = cnt;
  }
  *total = sum;
  return DLLM_OK;
}

dllm_status do_step(dllm_state* s, int j, const SelectRule& rule, int mode, int32_t* committed, int* total,
                    cudaEvent_t e0 = nullptr, cudaEvent_t e1 = nullptr, bool commit_prev = false) {
  CKS(step_enqueue(s, j, rule, mode, commit_prev, false, 0, e0, e1));
  return step_collect(s, j, rule, 0, committed, total);
}

}  // namespace

extern "C" dllm_status dllm_prefill_refresh(dllm_state* s) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  return do_refresh(s);
}

extern "C" dllm_status dllm_denoise_step_ex(dllm_state* s, int32_t block_idx, const dllm_select* sel,
                                           int32_t cache_mode, int32_t* committed) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  SelectRule r;
  CKS(to_rule(sel, &r));
  int total = 0;
  return do_step(s, block_idx, r, cache_mode, committed, &total);
}

extern "C" int32_t dllm_denoise_step(dllm_state* s, int32_t block_idx, float tau, int32_t cache_mode,
                                     int32_t* committed) {
  if (!s) {
    set_error("NULL state");
    return -DLLM_EINVAL;
  }
  dllm_select sel{DLLM_SEL_THRESHOLD, tau, 1, 1.0f};
  SelectRule r;
  dllm_status st = to_rule(&sel, &r);
  if (st != DLLM_OK) return -(int32_t)st;
  int total = 0;
  st = do_step(s, block_idx, r, cache_mode, committed, &total);
  return st == DLLM_OK ? total : -(int32_t)st;
}

extern "C" dllm_status dllm_run(dllm_state* s, const dllm_select* sel, int32_t cache_mode, int32_t refresh_interval,
                                dllm_stats* stats) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  SelectRule r;
  CKS(to_rule(sel, &r));
  if (cache_mode < 0 || cache_mode > 2 || refresh_interval < 0) {
    set_error("bad cache mode %d or refresh interval %d", cache_mode, refresh_interval);
    return DLLM_EINVAL;
  }
  const auto t0 = std::chrono::steady_clock::now();
  const long long launches0 = s->launches;
  double refresh_ms = 0, step_ms = 0;
  int steps = 0, refreshes = 0, max_spb = 0, fused = 0;
  long long committed = 0, active = 0;
  const bool cached = cache_mode != DLLM_CACHE_NONE;
  // Under the bidirectional mask a refresh is deferred to the step after it
  // and both run as one no-cache forward of that step: the forward rewrites
  // every layer's K/V from the current canvas (the refresh), and a cached step
  // right after a refresh reads exactly those K/V for every key, so its block
  // rows are the step's.  The refresh's own forward stops after the last
  // layer's K/V; the fused one finishes the last layer and the LM head, which
  // costs far less than a separate step.  Under the block-causal mask the
  // same holds for the prefill and a refresh interval's refreshes (full
  // forwards under the mask); its block-boundary refreshes are commit
  // forwards over one block (below) and stay separate.
  const bool fuse = cached && s->fuse_refresh;
  bool pending = false;
  int pending_j = 0, pending_spb = 0;
  // Block-causal: block j's commit forward is deferred to block j+1's first
  // step when both fit one persistent launch (2B rows): one forward over the
  // two blocks writes block j's K/V from the final canvas and runs block
  // j+1's step, whose rows see block j's fresh K/V in the same layer.
  bool pending_commit = false;
  int commit_j = 0, commit_spb = 0;
  std::vector<int32_t> cnt(s->b);
  // the observer sees each event after it completed; a nonzero answer stops the run
  auto notify = [&](int event, int j, int spb) -> dllm_status {
    if (s->hook && s->hook(s->hook_user, event, j, spb) != 0) {
      set_error("the run hook stopped the run at event %d (block %d, step %d of the block)", event, j, spb);
      return DLLM_ECANCELLED;
    }
    return DLLM_OK;
  };
  auto timed_refresh = [&]() -> dllm_status {
    CKS(do_refresh(s, s->ev_a, s->ev_b));
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, s->ev_a, s->ev_b));
    refresh_ms += ms;
    ++refreshes;
    return DLLM_OK;
  };
  auto refresh_before_step = [&](int j, int spb) -> dllm_status {
    if (fuse) {
      pending = true;
      pending_j = j;
      pending_spb = spb;
      return DLLM_OK;
    }
    CKS(timed_refresh());
    return notify(DLLM_EVENT_REFRESH, j, spb);
  };
  // Run-ahead: a block's next plain DualCache step is enqueued before the
  // current step's commits are read back, so that the GPU does not idle for
  // the host's round trip between steps.  When the current step finishes the
  // block, the step launched ahead finds no MASK in it and ends at once.
  // Off while a hook, per-kernel timing, the phase timeline or the trace
  // observe the run step by step; the trajectory is the same either way.
  const bool ahead_ok = s->run_ahead && !s->hook && !s->timing && !s->timeline && !s->trace &&
                        cache_mode == DLLM_CACHE_DUAL;
  auto rule_at = [&](int spb) {
    SelectRule rs = r;
    if (r.policy == 4) rs.k = std::max(1, r.k - spb);   // steps left in this block
    return rs;
  };
  // an error with a step still in flight: let it finish before returning
  auto drained = [&](dllm_status st) {
    if (st != DLLM_OK) cudaStreamSynchronize(s->st);
    return st;
  };
  cudaEvent_t ev0[2] = {s->ev_a, s->ev_c}, ev1[2] = {s->ev_b, s->ev_d};
  if (cached && s->n_blocks > 0) CKS(refresh_before_step(0, 0));
  for (int j = 0; j < s->n_blocks; ++j) {
    int spb = 0;
    int cur = 0;          // host slot of the step collected next
    bool ahead = false;   // step spb is already enqueued (launched ahead)
    for (;;) {
      int any = 0, act = 0;
      for (int i = 0; i < s->b; ++i) {
        const int rem = s->remaining[(size_t)i * s->n_blocks + j];
        any |= rem > 0;
        act += rem > 0;
      }
      if (!any) {
        if (ahead) {   // launched ahead of the block's last step: it found no MASK and did nothing
          int none = 0;
          CKS(drained(step_collect(s, j, rule_at(spb), cur, cnt.data(), &none)));
        }
        break;
      }
      const SelectRule rs = rule_at(spb);
      bool fused_step = false, commit_step = false;
      if (ahead) {
        ahead = false;   // a plain step, enqueued by the previous round
      } else {
        if (cached && refresh_interval > 0 && spb > 0 && spb % refresh_interval == 0) CKS(refresh_before_step(j, spb));
        fused_step = pending;
        commit_step = pending_commit;
        s->fused_fwd = fused_step;
        const dllm_status st = step_enqueue(s, j, rs, fused_step ? (int)DLLM_CACHE_NONE : cache_mode, commit_step,
                                            false, cur, ev0[cur], ev1[cur]);
        s->fused_fwd = false;
        CKS(drained(st));
      }
      const int nx = spb + 1;
      if (ahead_ok && !(cached && refresh_interval > 0 && nx % refresh_interval == 0) &&
          use_persistent(s, SK_DUAL, j)) {
        CKS(drained(step_enqueue(s, j, rule_at(nx), cache_mode, false, true, cur ^ 1, ev0[cur ^ 1], ev1[cur ^ 1])));
        ahead = true;
      }
      int total = 0;
      CKS(drained(step_collect(s, j, rs, cur, cnt.data(), &total)));
      float ms = 0;
      CK(cudaEventElapsedTime(&ms, ev0[cur], ev1[cur]));
      if (ahead) cur ^= 1;
      if (fused_step || commit_step) {
        refresh_ms += ms;
        ++refreshes;
        ++fused;
        if (fused_step) CKS(notify(DLLM_EVENT_REFRESH, pending_j, pending_spb));
        if (commit_step) CKS(notify(DLLM_EVENT_COMMIT_FORWARD, commit_j, commit_spb));
        pending = false;
        pending_commit = false;
      } else {
        step_ms += ms;
      }
      ++steps;
      ++spb;
      committed += total;
      active += act;
      CKS(notify(DLLM_EVENT_STEP, j, spb - 1));
    }
    max_spb = std::max(max_spb, spb);
    if (cached && j + 1 < s->n_blocks) {
      if (s->block_causal && s->fuse_refresh && cache_mode == DLLM_CACHE_DUAL && use_persistent(s, SK_COMMIT, j + 1)) {
        pending_commit = true;
        commit_j = j;
        commit_spb = spb;
      } else if (s->block_causal) {
        // nothing earlier attends to a later block: caching the finished
        // block's own K/V (one block forward) makes the cache exact again
        CK(cudaEventRecord(s->ev_a, s->st));
        CK(cudaMemsetAsync(s->count_err + s->b, 0, 4, s->st));
        SelectRule none{0, 2.0f, 1, 1.0f};
        const int blk = s->P + j * s->B;
        CKS(run_forward(s, blk, s->B, true, blk, none));
        CK(cudaEventRecord(s->ev_b, s->st));
        CKS(finish_sync(s));
        float ms = 0;
        CK(cudaEventElapsedTime(&ms, s->ev_a, s->ev_b));
        refresh_ms += ms;
        ++refreshes;
        CKS(notify(DLLM_EVENT_COMMIT_FORWARD, j, spb));
      } else {
        CKS(refresh_before_step(j, spb));
      }
    }
  }
  if (pending) {   // no step followed the last refresh
    CKS(timed_refresh());
    CKS(notify(DLLM_EVENT_REFRESH, pending_j, pending_spb));
  }
  if (stats) {
    stats->wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    stats->refresh_ms = refresh_ms;
    stats->step_ms = step_ms;
    stats->steps = steps;
    stats->refreshes = refreshes;
    stats->blocks = s->n_blocks;
    stats->max_steps_per_block = max_spb;
    stats->committed = committed;
    stats->tau_bar = active > 0 ? (double)committed / (double)active : 0.0;
    stats->kernel_launches = s->launches - launches0;
    stats->fused_steps = fused;
    stats->reserved = 0;
  }
  return DLLM_OK;
}

extern "C" dllm_status dllm_generate(dllm_model* m, const int32_t* prompts, int32_t b, int32_t P, int32_t gen_len,
                                     int32_t block, float tau, int32_t cache_mode, int32_t* out_tokens,
                                     dllm_stats* stats) {
  if (!m || (!prompts && P > 0) || !out_tokens) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  const auto t0 = std::chrono::steady_clock::now();
  dllm_state* s = nullptr;
  std::vector<int32_t> empty;
  CKS(dllm_state_create(m, prompts ? prompts : empty.data(), b, P, gen_len, block, nullptr, &s));
  dllm_select sel{DLLM_SEL_THRESHOLD, tau, 1, 1.0f};
  dllm_status st = dllm_run(s, &sel, cache_mode, 0, stats);
  if (st == DLLM_OK && gen_len > 0) {
    cudaError_t e = cudaMemcpy2DAsync(out_tokens, (size_t)gen_len * 4, s->x + P, (size_t)s->T * 4,
                                      (size_t)gen_len * 4, b, cudaMemcpyDeviceToHost, s->st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s->st);
    if (e != cudaSuccess) {
      set_error("copying the answer back failed: %s", cudaGetErrorString(e));
      st = DLLM_ECUDA;
    }
  }
  dllm_free_state(s);
  if (stats && st == DLLM_OK)
    stats->wall_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  return st;
}

extern "C" dllm_status dllm_read_state(const dllm_state* s, int32_t* tokens, float* conf, int32_t* arg) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  CK(cudaStreamSynchronize(s->st));
  if (tokens) CK(cudaMemcpy(tokens, s->x, (size_t)s->b * s->T * 4, cudaMemcpyDeviceToHost));
  if (conf) CK(cudaMemcpy(conf, s->conf, (size_t)s->b * s->B * 4, cudaMemcpyDeviceToHost));
  if (arg) CK(cudaMemcpy(arg, s->arg, (size_t)s->b * s->B * 4, cudaMemcpyDeviceToHost));
  return DLLM_OK;
}

extern "C" dllm_status dllm_read_hidden(const dllm_state* s, float* h) {
  if (!s || !h) {
    set_error("NULL argument");
    return DLLM_EINVAL;
  }
  const int d = s->m->cfg.d_model;
  CK(cudaStreamSynchronize(s->st));
  const int off = s->last_blk - s->last_row0;
  if (off < 0 || off + s->B > s->last_R) {
    set_error("no denoise step has run");
    return DLLM_ESTATE;
  }
  for (int i = 0; i < s->b; ++i)
    CK(cudaMemcpy(h + (size_t)i * s->B * d, s->h + ((size_t)i * s->last_R + off) * d, (size_t)s->B * d * 4,
                  cudaMemcpyDeviceToHost));
  return DLLM_OK;
}

extern "C" dllm_status dllm_read_kv(const dllm_state* s, int32_t layer, float* k, float* v) {
  if (!s || layer < 0 || layer >= s->m->cfg.n_layers) {
    set_error("bad argument");
    return DLLM_EINVAL;
  }
  const dllm_config& c = s->m->cfg;
  const size_t plane = (size_t)s->b * c.n_heads * s->T * c.head_dim;
  std::vector<uint16_t> hi(plane), lo(plane);
  CK(cudaStreamSynchronize(s->st));
  for (int kvi = 0; kvi < 2; ++kvi) {
    float* dst = kvi == 0 ? k : v;
    if (!dst) continue;
    const uint16_t* src = s->kv + ((size_t)layer * 2 + kvi) * 2 * plane;
    CK(cudaMemcpy(hi.data(), src, plane * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(lo.data(), src + plane, plane * 2, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < plane; ++i) {
      const uint32_t uh = (uint32_t)hi[i] << 16, ul = (uint32_t)lo[i] << 16;
      float fh, fl;
      std::memcpy(&fh, &uh, 4);
      std::memcpy(&fl, &ul, 4);
      dst[i] = s->split ? fh + fl : fh;
    }
  }
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_precision(dllm_state* s, int32_t mode) {
  if (!s || (mode != DLLM_PREC_SPLIT && mode != DLLM_PREC_BF16)) {
    set_error("bad precision mode %d", mode);
    return DLLM_EINVAL;
  }
  s->split = mode == DLLM_PREC_SPLIT;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_mask(dllm_state* s, int32_t mask) {
  if (!s || (mask != DLLM_MASK_BIDIRECTIONAL && mask != DLLM_MASK_BLOCK_CAUSAL)) {
    set_error("bad attention mask %d", mask);
    return DLLM_EINVAL;
  }
  s->block_causal = mask == DLLM_MASK_BLOCK_CAUSAL;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_persistent(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->persistent = enable != 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_fused_refresh(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->fuse_refresh = enable != 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_run_ahead(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->run_ahead = enable != 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_step_timeline(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->timeline = enable != 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_read_step_timeline(const dllm_state* s, uint64_t* out, int64_t capacity, int32_t* ctas,
                                               int32_t* phases) {
  if (!s || !s->d_timeline) {
    set_error("no persistent-step timeline was recorded");
    return DLLM_ESTATE;
  }
  const size_t n = (size_t)s->m->sms * s->n_phases * kTimelineSlots;
  if (ctas) *ctas = s->m->sms;
  if (phases) *phases = s->n_phases;
  if (!out) return DLLM_OK;
  if ((size_t)capacity < n) {
    set_error("timeline needs %zu values", n);
    return DLLM_EINVAL;
  }
  CK(cudaStreamSynchronize(s->st));
  CK(cudaMemcpy(out, s->d_timeline, n * 8, cudaMemcpyDeviceToHost));
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_run_hook(dllm_state* s, dllm_run_hook hook, void* user) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->hook = hook;
  s->hook_user = user;
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_trace(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  if (enable && !s->trace_buf) {
    const size_t n = (size_t)(s->m->cfg.n_layers + 1) * s->b * s->T * s->m->cfg.d_model * 4;
    CKS(dev_alloc((void**)&s->trace_buf, n));
  }
  s->trace = enable != 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_read_trace(const dllm_state* s, float* out, int64_t capacity, int32_t* rows_per_seq,
                                       int32_t* first_pos) {
  if (!s || !s->trace_buf) {
    set_error("tracing was never enabled");
    return DLLM_ESTATE;
  }
  const size_t n = (size_t)s->b * s->last_R * s->m->cfg.d_model;
  const size_t need = (size_t)(s->m->cfg.n_layers + 1) * n;
  if (rows_per_seq) *rows_per_seq = s->last_R;
  if (first_pos) *first_pos = s->last_row0;
  if (!out) return DLLM_OK;
  if ((size_t)capacity < need) {
    set_error("trace needs %zu floats, capacity %lld", need, (long long)capacity);
    return DLLM_EINVAL;
  }
  CK(cudaStreamSynchronize(s->st));
  CK(cudaMemcpy(out, s->trace_buf, need * 4, cudaMemcpyDeviceToHost));
  return DLLM_OK;
}

extern "C" dllm_status dllm_state_set_kernel_timing(dllm_state* s, int32_t enable) {
  if (!s) {
    set_error("NULL state");
    return DLLM_EINVAL;
  }
  s->timing = enable != 0;
  for (int i = 0; i < KC_N; ++i) {
    s->kt_ms[i] = 0;
    s->kt_n[i] = 0;
    s->kt_bytes[i] = 0;
  }
  s->pending.clear();
  s->ev_next = 0;
  return DLLM_OK;
}

extern "C" dllm_status dllm_kernel_times(const dllm_state* s, double* ms, int64_t* launches, double* bytes,
                                         int32_t n) {
  if (!s || n < 0) {
    set_error("bad argument");
    return DLLM_EINVAL;
  }
  for (int i = 0; i < n && i < KC_N; ++i) {
    if (ms) ms[i] = s->kt_ms[i];
    if (launches) launches[i] = s->kt_n[i];
    if (bytes) bytes[i] = s->kt_bytes[i];
  }
  return DLLM_OK;
}

// ====================================================================== kernel-level ops
namespace {

struct OpWorkspace {
  float* ws = nullptr;
  int* cnt = nullptr;
  size_t cnt_n = 0;
  float* attn = nullptr;
  size_t attn_floats = 0;
  int* attn_cnt = nullptr;
  size_t attn_cnt_n = 0;
  int* err = nullptr;
};

std::mutex g_op_mu;
std::map<int, OpWorkspace> g_op_ws;

dllm_status op_workspace(OpWorkspace** out, size_t cnt_n, size_t attn_floats, size_t attn_cnt_n) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  OpWorkspace& w = g_op_ws[dev];
  if (!w.ws) {
    CKS(dev_alloc((void**)&w.ws, (size_t)device_sms() * 2 * 256 * 128 * 4));
    CKS(dev_alloc((void**)&w.err, 256));
    CK(cudaMemset(w.err, 0, 256));
  }
  if (w.cnt_n < cnt_n) {
    if (w.cnt) cudaFree(w.cnt);
    w.cnt = nullptr;
    CKS(dev_alloc((void**)&w.cnt, cnt_n * 4));
    CK(cudaMemset(w.cnt, 0, cnt_n * 4));
    w.cnt_n = cnt_n;
  }
  if (w.attn_floats < attn_floats) {
    if (w.attn) cudaFree(w.attn);
    w.attn = nullptr;
    CKS(dev_alloc((void**)&w.attn, attn_floats * 4));
    w.attn_floats = attn_floats;
  }
  if (w.attn_cnt_n < attn_cnt_n) {
    if (w.attn_cnt) cudaFree(w.attn_cnt);
    w.attn_cnt = nullptr;
    CKS(dev_alloc((void**)&w.attn_cnt, attn_cnt_n * 4));
    CK(cudaMemset(w.attn_cnt, 0, attn_cnt_n * 4));
    w.attn_cnt_n = attn_cnt_n;
  }
  *out = &w;
  return DLLM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" dllm_status dllm_op_gemm_trace(const uint16_t* W, const uint16_t* X, const uint16_t* X_lo, float* Y,
                                          int32_t M, int32_t N, int32_t K, uint64_t* trace, int32_t* grid_out,
                                          void* stream);

extern "C" dllm_status dllm_op_gemm(const uint16_t* W, const uint16_t* X, const uint16_t* X_lo, float* Y, int32_t M,
                                    int32_t N, int32_t K, void* stream) {
  return dllm_op_gemm_trace(W, X, X_lo, Y, M, N, K, nullptr, nullptr, stream);
}

extern "C" dllm_status dllm_op_gemm_trace(const uint16_t* W, const uint16_t* X, const uint16_t* X_lo, float* Y,
                                          int32_t M, int32_t N, int32_t K, uint64_t* trace, int32_t* grid_out,
                                          void* stream) {
  if (!W || !X || !Y || M < 1 || N < 1 || K < 8 || K % 8 != 0 || !aligned16(W) || !aligned16(X) ||
      (X_lo && !aligned16(X_lo))) {
    set_error("bad gemm arguments: M=%d N=%d K=%d (K %% 8 == 0, 16-byte aligned operands)", M, N, K);
    return DLLM_EINVAL;
  }
  std::lock_guard<std::mutex> lk(g_op_mu);
  const int BN = pick_bn(N, X_lo != nullptr);
  GemmParams p = {};
  p.split = X_lo != nullptr;
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = ceil_div(M, 128);
  p.n_tiles = ceil_div(N, BN);
  p.kc = ceil_div(K, 64);
  p.total = (long long)p.m_tiles * p.n_tiles * p.kc;
  OpWorkspace* w = nullptr;
  CKS(op_workspace(&w, (size_t)p.m_tiles * p.n_tiles, 0, 0));
  p.ws = w->ws;
  p.counters = w->cnt;
  p.err = w->err;
  p.y = Y;
  p.ldy = M;
  p.trace = reinterpret_cast<unsigned long long*>(trace);
  CUtensorMap ta, tb, tbl;
  CKS(map_2d(&ta, W, K, M, 128));
  CKS(map_2d(&tb, X, K, N, BN));
  tbl = tb;
  if (X_lo) CKS(map_2d(&tbl, X_lo, K, N, BN));
  const int grid = (int)std::min<long long>(device_sms(), p.total);
  if (p.total * (grid + 1) >= (1LL << 31)) {   // the kernel's stream-K arithmetic is 32-bit
    set_error("GEMM of %lld chunks is too large", (long long)p.total);
    return DLLM_EINVAL;
  }
  if (grid_out) *grid_out = grid;
  CK(launch_gemm(GEMM_PLAIN, BN, ta, tb, tbl, p, grid, static_cast<cudaStream_t>(stream), false));
  return DLLM_OK;
}

extern "C" dllm_status dllm_op_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                         uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R, int32_t T,
                                         void* stream) {
  if (!q || !k_cache || !v_cache || !out || b < 1 || H < 1 || (hd != 64 && hd != 128) || R < 1 || T < 1 ||
      !aligned16(k_cache) || !aligned16(v_cache)) {
    set_error("bad attention arguments: b=%d H=%d hd=%d R=%d T=%d", b, H, hd, R, T);
    return DLLM_EINVAL;
  }
  std::lock_guard<std::mutex> lk(g_op_mu);
  const int sms = device_sms();
  AttnPlan a = plan_attention(b, H, R, T, sms);
  const int QT = 16 * a.wq;
  const size_t works = (size_t)b * H * a.q_tiles;
  OpWorkspace* w = nullptr;
  CKS(op_workspace(&w, 1, works * a.splits * QT * (hd + 2), works));
  CUtensorMap tk, tv;
  CKS(map_kv(&tk, k_cache, hd, T, (uint64_t)b * H, 64));
  CKS(map_kv(&tv, v_cache, hd, T, (uint64_t)b * H, 64));
  AttnParams p = {};
  p.q = q;
  p.o = out;
  p.o_lo = nullptr;
  p.R = R;
  p.b = b;
  p.H = H;
  p.T = T;
  p.z_k0 = 0;
  p.z_v0 = 0;
  p.q_tiles = a.q_tiles;
  p.splits = a.splits;
  p.kps = a.kps;
  p.scale_log2 = kLog2e / std::sqrt((float)hd);
  p.ws_o = w->attn;
  p.ws_ml = w->attn + works * a.splits * QT * hd;
  p.counters = w->attn_cnt;
  p.err = w->err;
  CK(launch_attention(hd, a.wq, 64, tk, tv, p, dim3(a.splits, a.q_tiles * H, b), static_cast<cudaStream_t>(stream),
                      false));
  return DLLM_OK;
}

extern "C" dllm_status dllm_op_attention_tc(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                            uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R, int32_t T,
                                            void* stream) {
  return dllm_op_attention_tc_ex(q, k_cache, v_cache, out, b, H, hd, R, T, 0, stream);
}

extern "C" dllm_status dllm_op_attention_tc_ex(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                               uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R, int32_t T,
                                               int32_t splits, void* stream) {
  if (!q || !k_cache || !v_cache || !out || b < 1 || H < 1 || (hd != 64 && hd != 128) || R < 1 || T < 1 ||
      splits < 0 || splits > 8 || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) {
    set_error("bad attention arguments: b=%d H=%d hd=%d R=%d T=%d splits=%d", b, H, hd, R, T, splits);
    return DLLM_EINVAL;
  }
  std::lock_guard<std::mutex> lk(g_op_mu);
  CUtensorMap tq, tk, tv;
  CKS(map_2d(&tq, q, (uint64_t)H * hd, (uint64_t)b * R, 128));
  CKS(map_kv(&tk, k_cache, hd, T, (uint64_t)b * H, 64));
  CKS(map_kv(&tv, v_cache, hd, T, (uint64_t)b * H, 64));
  AttnPlan at = plan_attention_tc(b, H, R, T, device_sms());
  if (splits > 0) {
    at.kps = ceil_div(ceil_div(T, 64), splits) * 64;
    at.splits = ceil_div(T, at.kps);
    at.n_whole = 0;
  }
  const long long items = (long long)b * H * at.q_tiles;
  const long long works = tc_split_items(at, items);
  OpWorkspace* w = nullptr;
  CKS(op_workspace(&w, 1, at.splits > 1 ? (size_t)works * at.splits * 128 * (hd + 2) : 0,
                   at.splits > 1 ? (size_t)works : 0));
  AttnParams p = {};
  p.q = q;
  p.o = out;
  p.R = R;
  p.b = b;
  p.H = H;
  p.T = T;
  p.q_tiles = at.q_tiles;
  p.splits = at.splits;
  p.kps = at.kps;
  p.n_whole = (int)at.n_whole;
  p.ws_o = w->attn;
  p.ws_ml = w->attn + works * at.splits * 128 * hd;
  p.counters = w->attn_cnt;
  p.scale_log2 = kLog2e / std::sqrt((float)hd);
  p.err = w->err;
  CK(launch_attention_tc(hd, tq, tq, tk, tv, p, dim3((unsigned)tc_ctas(at, items)), static_cast<cudaStream_t>(stream),
                         false));
  return DLLM_OK;
}

// ---------------------------------------------------------------- bounded-wait probe
namespace dllm {
// One thread waits, with the persistent step's own dataflow wait, until
// *flag >= need or limit_ns have passed; on expiry the wait records
// ERR_PROBE in err and the kernel returns.  Nothing else is in flight.
__global__ void wait_probe_kernel(const int* flag, int need, unsigned long long limit_ns, int* err) {
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    abort_s = 0;
    flag_wait_for(flag, need, &abort_s, err, limit_ns, ERR_PROBE);
  }
}
}  // namespace dllm

// ---------------------------------------------------------------- attention without allocation
// Scratch of dllm_op_attention_noalloc, in static storage of this library's
// module: the key-split partials (o, m, l) and the per-work merge counters.
// Module load zero-fills it; each work's last-arriving split puts its counter
// back to 0, and every call also clears the counters it uses before its
// launch.  The error word stays set until dllm_op_check reads it.
constexpr size_t kNoAllocAttnFloats = size_t(1) << 20;   // 4 MiB of split partials
constexpr int kNoAllocAttnWorks = 4096;                   // merge counters (b * H * query tiles)
static __device__ __align__(256) float g_noalloc_attn_ws[kNoAllocAttnFloats];
static __device__ __align__(256) int g_noalloc_attn_cnt[kNoAllocAttnWorks];
static __device__ __align__(256) int g_noalloc_attn_err[64];

namespace {

struct NoAllocScratch {
  float* ws;
  int* cnt;
  int* err;
};
constexpr int kNoAllocDevices = 64;
std::mutex g_noalloc_mu;
NoAllocScratch g_noalloc[kNoAllocDevices] = {};

// Device addresses of the static scratch for the current device, looked up
// once per device (cudaGetSymbolAddress with that device current).
dllm_status noalloc_scratch(NoAllocScratch* out) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocDevices) {
    set_error("device %d outside the %d devices the no-alloc scratch table holds", dev, kNoAllocDevices);
    return DLLM_EINVAL;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocScratch& s = g_noalloc[dev];
  if (!s.ws) {
    NoAllocScratch t = {};
    CK(cudaGetSymbolAddress(reinterpret_cast<void**>(&t.ws), g_noalloc_attn_ws));
    CK(cudaGetSymbolAddress(reinterpret_cast<void**>(&t.cnt), g_noalloc_attn_cnt));
    CK(cudaGetSymbolAddress(reinterpret_cast<void**>(&t.err), g_noalloc_attn_err));
    s = t;
  }
  *out = s;
  return DLLM_OK;
}

}  // namespace

extern "C" dllm_status dllm_op_attention_noalloc(const uint16_t* q, const uint16_t* k_cache,
                                                 const uint16_t* v_cache, uint16_t* out, int32_t b, int32_t H,
                                                 int32_t hd, int32_t R, int32_t T, void* stream) {
  if (!q || !k_cache || !v_cache || !out || b < 1 || H < 1 || (hd != 64 && hd != 128) || R < 1 || T < 1 ||
      !aligned16(k_cache) || !aligned16(v_cache)) {
    set_error("bad attention arguments: b=%d H=%d hd=%d R=%d T=%d", b, H, hd, R, T);
    return DLLM_EINVAL;
  }
  NoAllocScratch sc;
  CKS(noalloc_scratch(&sc));
  // the same plan as dllm_op_attention, so that both give identical outputs
  const AttnPlan a = plan_attention(b, H, R, T, device_sms());
  const int QT = 16 * a.wq;
  const size_t works = (size_t)b * H * a.q_tiles;
  const size_t floats = a.splits > 1 ? works * a.splits * QT * (hd + 2) : 0;
  if (floats > kNoAllocAttnFloats || (a.splits > 1 && works > (size_t)kNoAllocAttnWorks)) {
    set_error("attention b=%d H=%d hd=%d R=%d T=%d needs %zu scratch floats and %zu counters; the no-alloc "
              "variant holds %zu floats and %d counters (use dllm_op_attention)",
              b, H, hd, R, T, floats, works, kNoAllocAttnFloats, kNoAllocAttnWorks);
    return DLLM_EINVAL;
  }
  CUtensorMap tk, tv;
  CKS(map_kv(&tk, k_cache, hd, T, (uint64_t)b * H, 64));
  CKS(map_kv(&tv, v_cache, hd, T, (uint64_t)b * H, 64));
  // the merge counters this launch uses start at zero even if an earlier
  // launch gave up a bounded wait and left them counted (stream-ordered, no
  // allocation)
  if (a.splits > 1) CK(cudaMemsetAsync(sc.cnt, 0, works * sizeof(int), static_cast<cudaStream_t>(stream)));
  AttnParams p = {};
  p.q = q;
  p.o = out;
  p.o_lo = nullptr;
  p.R = R;
  p.b = b;
  p.H = H;
  p.T = T;
  p.z_k0 = 0;
  p.z_v0 = 0;
  p.q_tiles = a.q_tiles;
  p.splits = a.splits;
  p.kps = a.kps;
  p.scale_log2 = kLog2e / std::sqrt((float)hd);
  p.ws_o = sc.ws;
  p.ws_ml = sc.ws + works * a.splits * QT * hd;
  p.counters = sc.cnt;
  p.err = sc.err;
  CK(launch_attention(hd, a.wq, 64, tk, tv, p, dim3(a.splits, a.q_tiles * H, b), static_cast<cudaStream_t>(stream),
                      false));
  return DLLM_OK;
}

extern "C" dllm_status dllm_op_check(int32_t* site, void* stream) {
  int dev = 0;
  CK(cudaGetDevice(&dev));
  int words[2] = {0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  OpWorkspace* w = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_op_mu);
    auto it = g_op_ws.find(dev);
    if (it != g_op_ws.end() && it->second.err) w = &it->second;
  }
  NoAllocScratch sc;
  CKS(noalloc_scratch(&sc));
  if (w) CK(cudaMemcpyAsync(&words[0], w->err, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaMemcpyAsync(&words[1], sc.err, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  if (w) CK(cudaMemsetAsync(w->err, 0, 4, st));
  CK(cudaMemsetAsync(sc.err, 0, 4, st));
  CK(cudaStreamSynchronize(st));
  const int code = words[0] ? words[0] : words[1];
  if (site) *site = code;
  if (code != 0) {
    set_error("a kernel-level call gave up a bounded wait (site %d)", code);
    return DLLM_ETIMEOUT;
  }
  return DLLM_OK;
}

extern "C" dllm_status dllm_op_wait_probe(const int32_t* flag, int32_t need, int32_t limit_us, void* stream) {
  if (!flag || limit_us < 1 || limit_us > 2000000 || (reinterpret_cast<uintptr_t>(flag) & 3) != 0) {
    set_error("bad wait probe arguments: limit_us=%d (1 .. 2000000), flag 4-byte aligned", limit_us);
    return DLLM_EINVAL;
  }
  OpWorkspace* w = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_op_mu);
    CKS(op_workspace(&w, 1, 0, 0));
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  wait_probe_kernel<<<1, 32, 0, st>>>(flag, need, (unsigned long long)limit_us * 1000ull, w->err);
  CK(cudaGetLastError());
  int32_t site = 0;
  return dllm_op_check(&site, stream);
}

extern "C" dllm_status dllm_op_select_commit(const float* conf, const int32_t* arg, int32_t* x, int32_t b, int32_t T,
                                             int32_t blk_start, int32_t B, int32_t mask_id, const dllm_select* sel,
                                             int32_t* count, void* stream) {
  if (!conf || !arg || !x || !count || b < 1 || B < 1 || B > kMaxBlock || blk_start < 0 || blk_start + B > T) {
    set_error("bad select arguments: b=%d T=%d blk_start=%d B=%d", b, T, blk_start, B);
    return DLLM_EINVAL;
  }
  SelectRule r;
  CKS(to_rule(sel, &r));
  SelectParams p{conf, arg, x, count, T, blk_start, B, mask_id, r};
  select_kernel<<<b, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  CK(cudaGetLastError());
  return DLLM_OK;
}

// ====================================================================== staleness diagnostics
namespace {

// Cosine of each cached K/V row (hi + lo) with the same row of a fresh full
// forward: one warp per row of head_dim elements, lanes summing in a fixed
// order.  rows = L * 2 * b * H * T; parts = 2 when the low halves are kept.
__global__ void kv_cosine_kernel(const uint16_t* cached, const uint16_t* fresh, float* out, long long rows, int hd,
                                 long long part_rows, int parts) {
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // row -> (layer*2 + kind, rest): the hi plane block of that (layer, kind), then
  // the lo plane block part_rows rows later (the cache always has both)
  const long long lk = row / part_rows, rest = row - lk * part_rows;
  const long long hi_row = lk * 2 * part_rows + rest;
  float dot = 0.0f, nc = 0.0f, nf = 0.0f;
  for (int e = lane; e < hd; e += 32) {
    float c = __uint_as_float((uint32_t)cached[hi_row * hd + e] << 16);
    float f = __uint_as_float((uint32_t)fresh[hi_row * hd + e] << 16);
    if (parts == 2) {
      c += __uint_as_float((uint32_t)cached[(hi_row + part_rows) * hd + e] << 16);
      f += __uint_as_float((uint32_t)fresh[(hi_row + part_rows) * hd + e] << 16);
    }
    dot = fmaf(c, f, dot);
    nc = fmaf(c, c, nc);
    nf = fmaf(f, f, nf);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    dot += __shfl_xor_sync(0xffffffffu, dot, o);
    nc += __shfl_xor_sync(0xffffffffu, nc, o);
    nf += __shfl_xor_sync(0xffffffffu, nf, o);
  }
  if (lane == 0) out[row] = (nc > 0.0f && nf > 0.0f) ? dot / sqrtf(nc * nf) : 1.0f;
}

// The block forward (DualCache rows) on the current cache, predictions only:
// the canvas is restored afterwards.
dllm_status block_predict(dllm_state* s, int j, std::vector<float>& conf, std::vector<int32_t>& arg) {
  const int blk = s->P + j * s->B;
  const size_t nb = (size_t)s->b * s->T;
  CK(cudaMemcpyAsync(s->x_save, s->x, nb * 4, cudaMemcpyDeviceToDevice, s->st));
  CK(cudaMemsetAsync(s->count_err, 0, (s->b + 1) * 4, s->st));
  SelectRule keep_all{1, 0.0f, kMaxBlock, 1.0f};
  CKS(run_forward(s, blk, s->B, false, blk, keep_all));
  CKS(finish_sync(s));
  conf.resize((size_t)s->b * s->B);
  arg.resize((size_t)s->b * s->B);
  CK(cudaMemcpy(conf.data(), s->conf, conf.size() * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(arg.data(), s->arg, arg.size() * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpyAsync(s->x, s->x_save, nb * 4, cudaMemcpyDeviceToDevice, s->st));
  CK(cudaStreamSynchronize(s->st));
  return DLLM_OK;
}

}  // namespace

extern "C" dllm_status dllm_staleness(dllm_state* s, int32_t block_idx, float* k_cos, float* v_cos, float* agree,
                                      float* max_dconf) {
  if (!s || block_idx < 0 || block_idx >= s->n_blocks || !k_cos || !v_cos || !agree || !max_dconf) {
    set_error("bad staleness arguments (block %d)", block_idx);
    return DLLM_EINVAL;
  }
  const dllm_config& c = s->m->cfg;
  const int L = c.n_layers, H = c.n_heads, hd = c.head_dim;
  const size_t plane = (size_t)s->b * H * s->T * hd;          // elements of one (layer, kind, part) block
  const size_t kv_elems = (size_t)L * 4 * plane;
  const long long rows = (long long)L * 2 * s->b * H * s->T;
  if (!s->kv_fresh) {
    CKS(dev_alloc((void**)&s->kv_fresh, kv_elems * 2));
    CKS(dev_alloc((void**)&s->x_save, (size_t)s->b * s->T * 4));
    CKS(dev_alloc((void**)&s->row_cos, (size_t)rows * 4));
    CKS(map_kv(&s->tm_kv_fresh, s->kv_fresh, hd, s->T, (uint64_t)L * 4 * s->b * H, kStateAttnKT));
  }
  // the cache's own prediction for block j
  std::vector<float> conf_c, conf_f;
  std::vector<int32_t> arg_c, arg_f;
  CKS(block_predict(s, block_idx, conf_c, arg_c));
  // a fresh full forward over the current canvas into the scratch K/V, and
  // the block's prediction from it (= the prediction without a cache)
  std::swap(s->kv, s->kv_fresh);
  std::swap(s->tm_kv, s->tm_kv_fresh);
  dllm_status st = DLLM_OK;
  {
    SelectRule none{0, 2.0f, 1, 1.0f};
    CK(cudaMemsetAsync(s->count_err, 0, (s->b + 1) * 4, s->st));
    st = run_forward(s, 0, s->T, true, 0, none);
    if (st == DLLM_OK) st = finish_sync(s);
    if (st == DLLM_OK) st = block_predict(s, block_idx, conf_f, arg_f);
  }
  std::swap(s->kv, s->kv_fresh);
  std::swap(s->tm_kv, s->tm_kv_fresh);
  CKS(st);
  // cosines of cached and fresh rows; the fresh block rows were recomputed by
  // the block forward into the scratch, so they match the block step's
  const int parts = s->split ? 2 : 1;
  const long long part_rows = (long long)s->b * H * s->T;
  const int warps = 8;
  kv_cosine_kernel<<<(unsigned)((rows + warps - 1) / warps), warps * 32, 0, s->st>>>(
      s->kv, s->kv_fresh, s->row_cos, rows, hd, part_rows, parts);
  CK(cudaGetLastError());
  std::vector<float> cosv((size_t)rows);
  CK(cudaMemcpyAsync(cosv.data(), s->row_cos, cosv.size() * 4, cudaMemcpyDeviceToHost, s->st));
  CK(cudaStreamSynchronize(s->st));
  const int blk = s->P + block_idx * s->B;
  for (int l = 0; l < L; ++l) {
    for (int kind = 0; kind < 2; ++kind) {
      double sum = 0.0;
      long long n = 0;
      for (int i = 0; i < s->b; ++i)
        for (int h = 0; h < H; ++h)
          for (int t = 0; t < s->T; ++t) {
            if (t >= blk && t < blk + s->B) continue;   // the block's own rows are recomputed every step
            sum += cosv[(((size_t)(l * 2 + kind) * s->b + i) * H + h) * s->T + t];
            ++n;
          }
      (kind == 0 ? k_cos : v_cos)[l] = n ? (float)(sum / n) : 1.0f;
    }
  }
  // agreement at the block's MASK positions
  std::vector<int32_t> x((size_t)s->b * s->T);
  CK(cudaMemcpy(x.data(), s->x, x.size() * 4, cudaMemcpyDeviceToHost));
  long long same = 0, total = 0;
  float dmax = 0.0f;
  for (int i = 0; i < s->b; ++i)
    for (int k = 0; k < s->B; ++k) {
      if (x[(size_t)i * s->T + blk + k] != c.vocab) continue;
      const size_t o = (size_t)i * s->B + k;
      same += arg_c[o] == arg_f[o];
      ++total;
      dmax = std::max(dmax, std::fabs(conf_c[o] - conf_f[o]));
    }
  *agree = total ? (float)same / (float)total : 1.0f;
  *max_dconf = dmax;
  return DLLM_OK;
}

// ====================================================================== misc
extern "C" const char* dllm_last_error(void) { return g_err; }

extern "C" const char* dllm_status_string(int32_t st) {
  switch (st) {
    case DLLM_OK: return "ok";
    case DLLM_EINVAL: return "invalid argument";
    case DLLM_ENOMEM: return "out of memory";
    case DLLM_ECUDA: return "CUDA error";
    case DLLM_EIO: return "I/O error";
    case DLLM_ESTATE: return "invalid state";
    case DLLM_ETIMEOUT: return "kernel wait timed out";
    case DLLM_ECANCELLED: return "stopped by the run hook";
    default: return "unknown status";
  }
}

extern "C" int32_t dllm_version(void) { return 100; }
