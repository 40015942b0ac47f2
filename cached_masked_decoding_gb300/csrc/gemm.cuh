// Weight-streaming tensor-core GEMM with fused epilogues.
//
//   D[m][r] = sum_k W[m][k] * X[r][k]     (W: weights [M][K], X: activations [N][K], bf16)
//
// "Swap-AB" form: the weights are the 128-row A operand, the N activation rows
// the narrow B operand, so a denoise step with n = batch*block rows is one
// pass over the weights with n MACs per weight element.  One CTA per SM:
//   warp 0  TMA producer (A and B tiles into an smem ring, 128-byte swizzle),
//   warp 1  tcgen05.mma issuer (M=128, N=BN, K=16 per instruction, f32 in TMEM,
//           two TMEM accumulators so the epilogue of one tile overlaps the
//           main loop of the next),
//   warps 2-5  epilogue (tcgen05.ld, 32 columns at a time).
// Activation precision: with p.split the activations arrive as two bf16
// arrays, x = hi + lo (lo = bf16(x - hi), so the pair carries ~16 mantissa
// bits); both land in one B tile of 2*BN rows and one MMA of width 2*BN
// yields W.hi and W.lo side by side in TMEM, summed in the epilogue.  The
// weights are read once either way; while the GEMM is bound by HBM the extra
// MMA width is free.
// Work split: W = tiles / gridDim.x whole waves of tiles - CTA c takes tiles
// w*G + c, so CTAs side by side work on tiles side by side, which share their
// weight rows (tiles are numbered m-major): a weight tile comes from HBM once
// per wave and from L2 for the other n-tiles.  The remaining tiles' chunks of
// 64 reduction elements are cut into gridDim.x equal contiguous ranges
// ("stream-K"), so every SM streams the same number of bytes.  A tile cut
// between CTAs is finished by the last contributor to arrive, which sums every
// contributor's partial in contributor order: results do not depend on arrival
// order.  Each CTA runs its stream-K range before its whole tiles, so that the
// partials' exchange and the fix-up epilogues overlap the whole tiles' main
// loops instead of trailing the launch.
#pragma once

#include "ptx.cuh"

namespace dllm {

enum GemmKind : int { GEMM_PLAIN = 0, GEMM_QKV = 1, GEMM_RESID = 2, GEMM_SWIGLU = 3, GEMM_LMHEAD = 4 };

struct GemmParams {
  int M, N, K;            // weight rows, activation rows, reduction length
  int m_tiles, n_tiles, kc;
  long long total;        // m_tiles * n_tiles * kc
  float* ws;              // fix-up partials [grid][2][BN][128]
  int* counters;          // [m_tiles * n_tiles], zero between launches
  int* err;
  unsigned long long* trace;  // optional [grid][8] per-CTA timeline (diagnostics), or null
  int split;              // activations as a hi/lo bf16 pair (BN <= 128)
  // RMSNorm row factor of the activation rows: rsqrt(sum_t ss_in[r][t] * inv_d + eps)
  const float* ss_in;
  int ss_in_tiles;
  float inv_d, eps;
  // row r of X <-> sequence r / R, position row0 + r % R
  int R, row0;
  // GEMM_QKV
  uint16_t* q_out;        // [N][d]
  uint16_t* q_out_lo;     // low halves of q, or null (then K/V low halves are not written either)
  uint16_t* kv;           // cache [L][K|V][hi|lo][b][H][T_pad][hd]
  const float2* rope_cs;  // [T_pad][hd/2] (cos, sin)
  int d_model, head_dim, n_heads, T_pad, b_seqs, layer;
  // GEMM_RESID
  float* h;               // residual [N][d]
  const uint16_t* g_next; // next RMSNorm gain [d]
  uint16_t* xn_out;       // bf16(h * g_next) [rows][d]
  uint16_t* xn_out_lo;    // bf16(h * g_next - hi), or null
  float* ss_out;          // per-128-column sums of h^2 [rows][d/128]
  int remap;              // 1: output rows are the block rows (final layer)
  int blk_start, blk_len;
  // GEMM_SWIGLU
  uint16_t* act;          // [N][act_ld]
  uint16_t* act_lo;       // low halves, or null
  int act_ld;
  // GEMM_LMHEAD
  float* st_m;            // [m_tiles][N] tile max logit
  float* st_s;            // [m_tiles][N] tile sum exp(l - max)
  int* st_a;              // [m_tiles][N] tile argmax (lowest id)
  // GEMM_PLAIN
  float* y;
  int ldy;
};

template <int BN>
struct GemmCfg {
  static constexpr int B_ROWS = BN <= 128 ? 2 * BN : BN;   // room for the lo rows when BN <= 128
  static constexpr int A_BYTES = 128 * 64 * 2;
  static constexpr int B_BYTES = B_ROWS * 64 * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = STAGE_BYTES <= 24576 ? 8 : (STAGE_BYTES <= 32768 ? 6 : 4);
  static constexpr int TMEM_COLS = 2 * B_ROWS;   // two accumulators; 128..512, a power of two
  static constexpr int XCH_FLOATS = 128 * 33;
  static constexpr int RED_FLOATS = 4 * 32 * 3;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + XCH_FLOATS * 4 + 256 * 4 + RED_FLOATS * 4 +
                                    (2 * STAGES + 4) * 8 + 64;
};

// ---------------------------------------------------------------- standalone GEMM work list
// One segment: kc-chunk run [k0, k0 + len) of one tile; `whole` when it is the
// full reduction of the tile; rg0 is its first chunk in remainder-chunk space
// (stream-K part only).
struct GemmSeg {
  int m, n, tile, k0, len;
  bool whole;
  uint32_t rg0;
};

// The segments of one CTA: its stream-K range of the remainder, then its
// whole tiles (see the work split above).
struct GemmWork {
  uint32_t G, cta, kc, n_tiles, W, full, total_r, rs, re;
  __device__ __forceinline__ void init(uint32_t G_, uint32_t cta_, uint32_t tiles, uint32_t kc_, uint32_t n_tiles_) {
    G = G_;
    cta = cta_;
    kc = kc_;
    n_tiles = n_tiles_;
    W = tiles / G;
    full = W * G;
    total_r = (tiles - full) * kc;
    rs = total_r ? cta * total_r / G : 0;
    re = total_r ? (cta + 1) * total_r / G : 0;
  }
  __device__ __forceinline__ uint32_t chunks() const { return W * kc + (re - rs); }
};

struct GemmSegCursor {
  uint32_t w, g;
  __device__ __forceinline__ void init(const GemmWork& wk) {
    w = 0;
    g = wk.rs;
  }
  __device__ __forceinline__ bool next(const GemmWork& wk, GemmSeg& o) {
    uint32_t tile;
    if (g < wk.re) {
      const uint32_t rt = g / wk.kc, k = g - rt * wk.kc;
      const uint32_t len = (wk.kc - k < wk.re - g) ? wk.kc - k : wk.re - g;
      tile = wk.full + rt;
      o.k0 = (int)k;
      o.len = (int)len;
      o.whole = (k == 0) && (len == wk.kc);
      o.rg0 = g;
      g += len;
    } else if (w < wk.W) {
      tile = w * wk.G + wk.cta;
      ++w;
      o.k0 = 0;
      o.len = (int)wk.kc;
      o.whole = true;
      o.rg0 = 0;
    } else {
      return false;
    }
    o.tile = (int)tile;
    o.m = (int)(tile / wk.n_tiles);
    o.n = (int)(tile - (uint32_t)o.m * wk.n_tiles);
    return true;
  }
};

// ---------------------------------------------------------------- chunk positions
// Stream-K bookkeeping in 32-bit integers (a phase has at most a few 1e5
// chunks, times the grid stays below 2^31) and without divisions in the
// per-chunk loops: 64-bit integer division is a long software sequence,
// and several of them per chunk would cap the TMA issue rate.
__device__ __forceinline__ uint32_t sk_begin(uint32_t cta, uint32_t G, uint32_t total) { return cta * total / G; }

// The CTA whose stream-K range holds chunk i.
__device__ __forceinline__ uint32_t sk_owner32(uint32_t i, uint32_t G, uint32_t total) {
  return ((i + 1) * G + total - 1) / total - 1;
}

// (k-chunk, n-tile, m-tile) of a chunk; chunks run k fastest, then n-tiles,
// then m-tiles.
struct ChunkPos {
  int k, n, m;
  __device__ __forceinline__ void init(uint32_t g, int kc, int n_tiles) {
    const uint32_t tile = g / (uint32_t)kc;
    k = (int)(g - tile * (uint32_t)kc);
    m = (int)(tile / (uint32_t)n_tiles);
    n = (int)(tile - (uint32_t)m * (uint32_t)n_tiles);
  }
  __device__ __forceinline__ void next(int kc, int n_tiles) {
    if (++k == kc) {
      k = 0;
      if (++n == n_tiles) {
        n = 0;
        ++m;
      }
    }
  }
};

// Slot and phase parity of a position in the shared-memory ring.
struct RingPos {
  int s;
  uint32_t par;
  __device__ __forceinline__ void next(int stages) {
    if (++s == stages) {
      s = 0;
      par ^= 1u;
    }
  }
};


// Sum over the 32 lanes of a warp of 32 per-lane columns: afterwards v[0] on
// lane c holds the total of column c.  Fixed pairing order (deterministic).
__device__ __forceinline__ void warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      float send = up ? v[i] : v[i + s];
      float keep = up ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
}

// Max with lowest-index tie-break, transposed like warp_transpose_sum.
__device__ __forceinline__ void warp_transpose_argmax(float (&v)[32], int (&id)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      float sv = up ? v[i] : v[i + s];
      int si = up ? id[i] : id[i + s];
      float kv = up ? v[i + s] : v[i];
      int ki = up ? id[i + s] : id[i];
      float rv = __shfl_xor_sync(0xffffffffu, sv, s);
      int ri = __shfl_xor_sync(0xffffffffu, si, s);
      const bool take = (rv > kv) || (rv == kv && ri < ki);
      v[i] = take ? rv : kv;
      id[i] = take ? ri : ki;
    }
  }
}

// Row stride (floats) of the [32 rows][128 features] staging of an epilogue
// tile in the exchange buffer: 16-byte aligned rows, 128 * 33 floats in all.
constexpr int kStageLd = 132;

// Eight floats as bf16 pairs: hi = bf16(x), lo = bf16(x - hi).
// A pair of floats as bf16 (x0 in the low half) and their bf16 residuals,
// with one paired conversion each (two scalar conversions cost a measurable
// part of an epilogue).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t*>(&b);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void split8v(const float (&f)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) split2(f[2 * t], f[2 * t + 1], h[t], l[t]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Eight consecutive floats (16-byte aligned) as bf16 pairs.
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  split8v(f, hi, lo);
}

// Epilogue of 32 consecutive activation rows (columns of the accumulator) for
// the thread's weight row m = m_idx*128 + l128.  v holds raw sums.  Every
// epilogue thread of the CTA calls this with the same (m_idx, r0).
// Each epilogue reads everything it needs first (parameters into registers,
// global loads as one batch, L2-coherent: other CTAs may have written the data
// earlier in the same launch), computes, then stores: a store between loads
// would force every later load to wait for it.
template <int KIND>
__device__ __forceinline__ void epi_chunk(const GemmParams& p, float (&v)[32], int m_idx, int r0, int l128,
                                          int lane, int q, float* xch, const float* rs, float* red,
                                          const float* h_pre = nullptr) {
  const int m = m_idx * 128 + l128;
  const int N = p.N;
  if constexpr (KIND == GEMM_PLAIN) {
    float* __restrict__ y = p.y;
    const int ldy = p.ldy, M = p.M;
    const bool scale = p.ss_in != nullptr;
    if (m < M) {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int r = r0 + c;
        if (r < N) y[(long long)r * ldy + m] = scale ? v[c] * rs[c] : v[c];
      }
    }
  } else if constexpr (KIND == GEMM_QKV) {
    const int d = p.d_model, hd = p.head_dim, half = hd >> 1;
    const int R = p.R, row0 = p.row0, T = p.T_pad, H = p.n_heads, layer = p.layer, b = p.b_seqs;
    const float2* __restrict__ rope = p.rope_cs;
    const int sec = (m_idx * 128) / d;          // uniform over the tile: 0 q, 1 k, 2 v
    const int mr = m - sec * d;
    const int j = mr % hd;
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] *= rs[c];
    if (sec < 2) {
      const int seq0 = r0 / R, i0 = r0 - seq0 * R;   // rows r0.. walk (seq, i) without dividing
      const int jj = j & (half - 1);
      float2 cs[32];
      int i = i0;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        cs[c] = __ldg(&rope[(long long)(row0 + i) * half + jj]);
        if (++i == R) i = 0;
      }
      named_bar_sync(1, 128);
#pragma unroll
      for (int c = 0; c < 32; ++c) xch[l128 * 33 + c] = v[c];
      named_bar_sync(1, 128);
      const int partner = l128 ^ half;
      const float sgn = (j < half) ? -1.0f : 1.0f;
      float pv[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pv[c] = xch[partner * 33 + c];
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = v[c] * cs[c].x + sgn * pv[c] * cs[c].y;
    }
    // Store through shared memory: the tile is staged as [32 rows][128
    // features] and written 8 features (16 bytes) per thread and store, not
    // one 2-byte element per thread and row.
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < 32; ++c) xch[c * kStageLd + l128] = v[c];
    named_bar_sync(1, 128);
    uint16_t* __restrict__ q_out = p.q_out;
    uint16_t* __restrict__ q_lo = p.q_out_lo;
    uint16_t* __restrict__ kv = p.kv;
    const int f0 = m_idx * 128 - sec * d;       // the tile's first feature within its section
#pragma unroll
    for (int e = l128; e < 32 * 16; e += 128) {
      const int row = e >> 4, f8 = (e & 15) * 8;
      const int r = r0 + row;
      if (r >= N) continue;
      uint4 hi, lo;
      split8(xch + row * kStageLd + f8, hi, lo);
      const int fm = f0 + f8;
      if (sec == 0) {
        *reinterpret_cast<uint4*>(&q_out[(long long)r * d + fm]) = hi;
        if (q_lo) *reinterpret_cast<uint4*>(&q_lo[(long long)r * d + fm]) = lo;
      } else {
        // one sequence needs no division; head_dim is 64 or 128
        const int seq = b == 1 ? 0 : r / R, i = r - seq * R;
        const int head = hd == 128 ? fm >> 7 : fm >> 6, jj = fm - head * hd;
        const long long plane = ((((long long)layer * 2 + (sec - 1)) * 2) * b + seq) * H + head;
        *reinterpret_cast<uint4*>(&kv[(plane * T + row0 + i) * hd + jj]) = hi;
        if (q_lo) *reinterpret_cast<uint4*>(&kv[((plane + (long long)b * H) * T + row0 + i) * hd + jj]) = lo;
      }
    }
  } else if constexpr (KIND == GEMM_RESID) {
    // Staged through shared memory as [32 rows][128 features]: warp q then
    // handles rows q, q+4, ..., lane handles features 4*lane .. 4*lane+3, so
    // every global access is a 16-byte (h) or 8-byte (bf16) vector and the
    // row's sum of squares is one warp reduction.
    const int d = p.d_model, R = p.R, row0 = p.row0, blk0 = p.blk_start, blen = p.blk_len;
    const bool remap = p.remap != 0;
    float* __restrict__ h = p.h;
    uint16_t* __restrict__ xo = p.xn_out;
    uint16_t* __restrict__ xl = p.xn_out_lo;
    float* __restrict__ sso = p.ss_out;
    const int fb = m_idx * 128 + lane * 4;
    const uint2 graw = __ldg(reinterpret_cast<const uint2*>(p.g_next + fb));
    float hv[8][4];
    if (h_pre) {
      // the rows r0.. were copied to h_pre ([32][128]) by this thread group's
      // asynchronous copies; the barrier below makes every thread's visible
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = r0 + q + 4 * k;
        const float4 x = r < N ? __ldcg(reinterpret_cast<const float4*>(&h[(long long)r * d + fb]))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        hv[k][0] = x.x;
        hv[k][1] = x.y;
        hv[k][2] = x.z;
        hv[k][3] = x.w;
      }
    }
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < 32; ++c) xch[c * kStageLd + l128] = v[c];
    named_bar_sync(1, 128);
    if (h_pre) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(h_pre + (q + 4 * k) * 128 + lane * 4);
        hv[k][0] = x.x;
        hv[k][1] = x.y;
        hv[k][2] = x.z;
        hv[k][3] = x.w;
      }
    }
    const float g4[4] = {__uint_as_float(graw.x << 16), __uint_as_float(graw.x & 0xffff0000u),
                         __uint_as_float(graw.y << 16), __uint_as_float(graw.y & 0xffff0000u)};
    // the eight rows' sums of squares are reduced across the warp together:
    // one dependent shuffle chain instead of eight (same order per row)
    float sqv[8];
    int rov[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = q + 4 * k;
      const int r = r0 + row;
      const float4 add = *reinterpret_cast<const float4*>(xch + row * kStageLd + lane * 4);
      hv[k][0] += add.x;
      hv[k][1] += add.y;
      hv[k][2] += add.z;
      hv[k][3] += add.w;
      int ro = r;
      if (remap) {
        const int seq = r / R, pos = row0 + r % R;
        const int bi = pos - blk0;
        ro = (bi >= 0 && bi < blen) ? seq * blen + bi : -1;
      }
      rov[k] = r < N ? ro : -1;
      float sq = 0.0f;
      if (r < N) {
        *reinterpret_cast<float4*>(&h[(long long)r * d + fb]) = make_float4(hv[k][0], hv[k][1], hv[k][2], hv[k][3]);
        if (ro >= 0) {
          uint32_t hb[2], lb[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) split2(hv[k][2 * t] * g4[2 * t], hv[k][2 * t + 1] * g4[2 * t + 1], hb[t], lb[t]);
          *reinterpret_cast<uint2*>(&xo[(long long)ro * d + fb]) = make_uint2(hb[0], hb[1]);
          if (xl) *reinterpret_cast<uint2*>(&xl[(long long)ro * d + fb]) = make_uint2(lb[0], lb[1]);
          sq = (hv[k][0] * hv[k][0] + hv[k][1] * hv[k][1]) + (hv[k][2] * hv[k][2] + hv[k][3] * hv[k][3]);
        }
      }
      sqv[k] = sq;
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1)
#pragma unroll
      for (int k = 0; k < 8; ++k) sqv[k] += __shfl_xor_sync(0xffffffffu, sqv[k], s);
    // lane k stores row q + 4k's sum
    float sq_out = sqv[0];
    int ro_out = rov[0];
#pragma unroll
    for (int k = 1; k < 8; ++k)
      if (lane == k) {
        sq_out = sqv[k];
        ro_out = rov[k];
      }
    if (lane < 8 && ro_out >= 0) sso[(long long)ro_out * (d >> 7) + m_idx] = sq_out;
  } else if constexpr (KIND == GEMM_SWIGLU) {
    // The tile's 128 weight rows are 64 gate rows then the 64 matching up
    // rows.  Staged as [feature][row]; then every thread forms 16 outputs of
    // one activation row, silu(gate) * up with the fast reciprocal (an IEEE
    // division here cost about 2 us per tile), and stores them as bf16 pairs.
    uint16_t* __restrict__ act = p.act;
    uint16_t* __restrict__ act_lo = p.act_lo;
    const int ld = p.act_ld;
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < 32; ++c) xch[l128 * 33 + c] = v[c] * rs[c];
    named_bar_sync(1, 128);
    const int row = l128 >> 2, j0 = (l128 & 3) * 16;
    const int r = r0 + row;
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float gt = xch[(j0 + i) * 33 + row], up = xch[(j0 + i + 64) * 33 + row];
      a[i] = __fdividef(gt, 1.0f + __expf(-gt)) * up;
    }
    if (r < N) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float f8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f8[i] = a[hf * 8 + i];
        uint4 hi, lo;
        split8v(f8, hi, lo);
        const long long o = (long long)r * ld + m_idx * 64 + j0 + hf * 8;
        *reinterpret_cast<uint4*>(&act[o]) = hi;
        if (act_lo) *reinterpret_cast<uint4*>(&act_lo[o]) = lo;
      }
    }
  } else if constexpr (KIND == GEMM_LMHEAD) {
    const int M = p.M;
    float lg[32];
    int id[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      lg[c] = (m < M) ? v[c] * rs[c] : -INFINITY;
      id[c] = m;
    }
    float mx[32];
    int ax[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) { mx[c] = lg[c]; ax[c] = id[c]; }
    warp_transpose_argmax(mx, ax, lane);
    // mx[0]/ax[0] on lane c: this warp's max / argmax of column c
    float e[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float mc = __shfl_sync(0xffffffffu, mx[0], c);
      e[c] = exp2f((lg[c] - mc) * kLog2e);
    }
    warp_transpose_sum(e, lane);
    named_bar_sync(1, 128);
    red[(q * 32 + lane) * 3 + 0] = mx[0];
    red[(q * 32 + lane) * 3 + 1] = e[0];
    red[(q * 32 + lane) * 3 + 2] = __int_as_float(ax[0]);
    named_bar_sync(1, 128);
    if (l128 < 32) {
      const int r = r0 + l128;
      if (r < N) {
        float Mx = red[(0 * 32 + l128) * 3 + 0];
        int A = __float_as_int(red[(0 * 32 + l128) * 3 + 2]);
#pragma unroll
        for (int w = 1; w < 4; ++w) {
          const float mw = red[(w * 32 + l128) * 3 + 0];
          if (mw > Mx) { Mx = mw; A = __float_as_int(red[(w * 32 + l128) * 3 + 2]); }
        }
        float S = 0.0f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float mw = red[(w * 32 + l128) * 3 + 0];
          const float sw = red[(w * 32 + l128) * 3 + 1];
          S += (mw == -INFINITY) ? 0.0f : sw * exp2f((mw - Mx) * kLog2e);
        }
        const long long o = (long long)m_idx * N + r;
        p.st_m[o] = Mx;
        p.st_s[o] = S;
        p.st_a[o] = A;
      }
    }
  }
}

// v += the low-half accumulator columns (BN + c0 ..) of the same rows.
template <int BN>
__device__ __forceinline__ void add_lo(uint32_t taddr, int c0, float (&v)[32]) {
  float w[32];
  tmem_ld32(taddr + (uint32_t)(BN + c0), w);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] += w[j];
}

template <int BN, int KIND>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmBlo, const GemmParams p) {
  using C = GemmCfg<BN>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  float* xch = reinterpret_cast<float*>(sB + STAGES * C::B_BYTES);
  float* rs_s = xch + C::XCH_FLOATS;
  float* red = rs_s + 256;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + C::RED_FLOATS);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bcast = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t G = gridDim.x, cta = blockIdx.x;
  const int kc = p.kc, n_tiles = p.n_tiles;
  GemmWork wk;
  wk.init(G, cta, (uint32_t)(p.m_tiles * n_tiles), (uint32_t)kc, (uint32_t)n_tiles);
  const bool split = BN <= 128 && p.split != 0;
  const int n_rows = split ? 2 * BN : BN;                      // MMA width
  const uint32_t stage_tx = (uint32_t)(C::A_BYTES + n_rows * 128);

  if (p.trace && threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    p.trace[cta * 8 + 0] = smid;
    p.trace[cta * 8 + 1] = globaltimer();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (p.split) prefetch_tensormap(&tmBlo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const int n = (int)wk.chunks();
      const int pre = n < STAGES ? n : STAGES;
      // weights do not depend on the previous kernel: start streaming them
      // before waiting for its activations
      GemmSegCursor sw;
      sw.init(wk);
      GemmSeg a;
      bool live = sw.next(wk, a);
      int ka = 0;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], stage_tx);
        tma_load_2d(sA + i * C::A_BYTES, &tmA, &full[i], (a.k0 + ka) * 64, a.m * 128, pol_w);
        if (++ka == a.len) {
          live = sw.next(wk, a);
          ka = 0;
        }
      }
      griddep_wait();
      {
        GemmSegCursor sx;
        sx.init(wk);
        GemmSeg x;
        sx.next(wk, x);
        int kx = 0;
        for (int i = 0; i < pre; ++i) {
          tma_load_2d(sB + i * C::B_BYTES, &tmB, &full[i], (x.k0 + kx) * 64, x.n * BN, pol_x);
          if (split) tma_load_2d(sB + i * C::B_BYTES + BN * 128, &tmBlo, &full[i], (x.k0 + kx) * 64, x.n * BN, pol_x);
          if (++kx == x.len) {
            sx.next(wk, x);
            kx = 0;
          }
        }
      }
      RingPos rw{pre % STAGES, (uint32_t)((pre / STAGES) & 1)};
      int issued = pre;
      for (int i = pre; i < n && live; ++i) {
        if (!mbar_wait(&empty[rw.s], rw.par ^ 1u, abort_flag, p.err, ERR_GEMM_EMPTY)) break;
        const int k = a.k0 + ka;
        mbar_arrive_expect_tx(&full[rw.s], stage_tx);
        tma_load_2d(sA + rw.s * C::A_BYTES, &tmA, &full[rw.s], k * 64, a.m * 128, pol_w);
        tma_load_2d(sB + rw.s * C::B_BYTES, &tmB, &full[rw.s], k * 64, a.n * BN, pol_x);
        if (split) tma_load_2d(sB + rw.s * C::B_BYTES + BN * 128, &tmBlo, &full[rw.s], k * 64, a.n * BN, pol_x);
        rw.next(STAGES);
        issued = i + 1;
        if (++ka == a.len) {
          live = sw.next(wk, a);
          ka = 0;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's smem goes away
        const int lo = issued > STAGES ? issued - STAGES : 0;
        for (int i = lo; i < issued; ++i)
          mbar_wait(&full[i % STAGES], (uint32_t)((i / STAGES) & 1), nullptr, p.err, ERR_GEMM_DRAIN);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16_f32(128, n_rows);
      RingPos rm{0, 0u};
      bool first = true;
      int seg = 0;
      bool ok = true;
      GemmSegCursor sc;
      sc.init(wk);
      GemmSeg sg;
      while (ok && sc.next(wk, sg)) {
        const int buf = seg & 1;
        const uint32_t use = (uint32_t)(seg >> 1);
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p.err, ERR_GEMM_TEMPTY)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * C::B_ROWS);
        for (int i = 0; i < sg.len; ++i) {
          if (!mbar_wait(&full[rm.s], rm.par, abort_flag, p.err, ERR_GEMM_FULL)) {
            ok = false;
            break;
          }
          if (p.trace && first) p.trace[cta * 8 + 2] = globaltimer();
          first = false;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + rm.s * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + rm.s * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc, (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[rm.s]);
          rm.next(STAGES);
        }
        if (!ok) break;
        mma_commit(&tfull[buf]);
        ++seg;
      }
      if (p.trace) p.trace[cta * 8 + 3] = globaltimer();
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    griddep_wait();
    const int q = warp & 3;
    const int l128 = q * 32 + lane;
    GemmSegCursor sc;
    sc.init(wk);
    GemmSeg sg;
    int seg = 0;
    int rs_tile = -1;
    while (sc.next(wk, sg)) {
      const bool full_tile = sg.whole;
      const int m_idx = sg.m;
      const int n_idx = sg.n;
      const int tile = sg.tile;
      const int buf = seg & 1;
      const uint32_t use = (uint32_t)(seg >> 1);

      if (n_idx != rs_tile) {
        // RMSNorm row factors of this activation tile.  One row per thread:
        // its partial sums of squares are contiguous, read as 16-byte vectors
        // in a single round of loads and summed in order.  (The tile order
        // changes the row tile at almost every tile, so this runs per tile;
        // staged through shared memory in four dependent rounds it had cost
        // ~17 us per tile in the refresh.)
        rs_tile = n_idx;
        named_bar_sync(1, 128);
        if (p.ss_in) {
          const int tiles = p.ss_in_tiles;
          for (int c = l128; c < BN; c += 128) {
            const int r = n_idx * BN + c;
            float sum = 0.0f;
            if (r < p.N) {
              const float* src = p.ss_in + (long long)r * tiles;
              if ((tiles & 3) == 0) {
                for (int t0 = 0; t0 < tiles; t0 += 32) {
                  const int nv = (tiles - t0) / 4 < 8 ? (tiles - t0) / 4 : 8;
                  float4 x[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j)
                    x[j] = j < nv ? __ldcg(reinterpret_cast<const float4*>(src + t0) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                  for (int j = 0; j < 8; ++j)
                    if (j < nv) sum = (((sum + x[j].x) + x[j].y) + x[j].z) + x[j].w;
                }
              } else {
                for (int t = 0; t < tiles; ++t) sum += __ldcg(&src[t]);
              }
            }
            rs_s[c] = r < p.N ? rsqrtf(sum * p.inv_d + p.eps) : 0.0f;
          }
        } else {
          for (int c = l128; c < BN; c += 128) rs_s[c] = 1.0f;
        }
        named_bar_sync(1, 128);
      }

      // every epilogue warp takes the same decision: a warp whose wait gave up
      // raised *abort_flag before this barrier
      mbar_wait(&tfull[buf], use & 1u, abort_flag, p.err, ERR_GEMM_TFULL);
      if (named_bar_or(1, 128, *abort_flag != 0)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::B_ROWS);
      if (full_tile) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)c0, v);
          if (split) add_lo<BN>(taddr, c0, v);
          if (c0 + 32 == BN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
          }
          epi_chunk<KIND>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red);
        }
      } else {
        const int slot = (sg.rg0 == wk.rs) ? 0 : 1;                // first segment of this CTA's stream-K range?
        float* wsp = p.ws + (((long long)cta * 2 + slot) * BN) * 128;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)c0, v);
          if (split) add_lo<BN>(taddr, c0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) __stcg(&wsp[(long long)(c0 + j) * 128 + l128], v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        named_bar_sync(1, 128);
        const uint32_t total = wk.total_r;                          // stream-K space: the remainder tiles
        const uint32_t t0 = sg.rg0 - (uint32_t)sg.k0;               // the tile's first chunk
        const uint32_t c_first = sk_owner32(t0, G, total), c_last = sk_owner32(t0 + (uint32_t)kc - 1, G, total);
        if (l128 == 0) {
          // contributors: the CTAs in [c_first, c_last] whose chunk range is not
          // empty (with fewer chunks than CTAs some ranges are)
          int contributors = 0;
          uint32_t st = sk_begin(c_first, G, total);
          for (uint32_t ctr = c_first; ctr <= c_last; ++ctr) {
            const uint32_t en = sk_begin(ctr + 1, G, total);
            contributors += st < en ? 1 : 0;
            st = en;
          }
          const int old = atomic_add_acq_rel_gpu(&p.counters[tile], 1);
          const int last = (old == contributors - 1);
          if (last) p.counters[tile] = 0;
          *bcast = last;
        }
        named_bar_sync(1, 128);
        if (*bcast) {
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 32) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
            // partials in contributor order, two at a time so that both sets
            // of loads are in flight together: ((v + p0) + p1) + ...
            uint32_t ctr = c_first;
            uint32_t st = sk_begin(c_first, G, total);
            while (ctr <= c_last) {
              const float* src0 = nullptr;
              const float* src1 = nullptr;
              int ns = 0;
              for (; ctr <= c_last && ns < 2; ++ctr) {
                const uint32_t en = sk_begin(ctr + 1, G, total);
                const uint32_t cst = st;
                st = en;
                if (cst == en) continue;                     // empty range: no partial
                const int sl = (cst >= t0) ? 0 : 1;          // its first segment starts in this tile?
                const float* sp = p.ws + (((long long)ctr * 2 + sl) * BN) * 128 + (long long)c0 * 128 + l128;
                if (ns == 0) src0 = sp;
                else src1 = sp;
                ++ns;
              }
              if (ns == 2) {
                float x0[32], x1[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  x0[j] = __ldcg(src0 + j * 128);
                  x1[j] = __ldcg(src1 + j * 128);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = (v[j] + x0[j]) + x1[j];
              } else if (ns == 1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += __ldcg(src0 + j * 128);
              }
            }
            epi_chunk<KIND>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red);
          }
        }
      }
      ++seg;
    }
    if (p.trace && l128 == 0) p.trace[cta * 8 + 4] = globaltimer();
  }
  // Lanes 1-31 of the producer and MMA warps skipped their roles and arrive
  // here first: reconverge each warp before the CTA-wide barrier (an aligned
  // barrier reached by part of a warp would let the warp count as arrived
  // while lane 0 still works, and tensor memory could be freed under the
  // epilogue warps' last reads).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (p.trace && threadIdx.x == 0) p.trace[cta * 8 + 5] = globaltimer();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace dllm
