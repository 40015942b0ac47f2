// Non-causal block attention over the K/V cache (the zhongzhuzhou.org notes,
// section 2, eq. 3, with every query reading every key: section 3, Algorithm
// 1 step 7 - fresh block K/V plus cached prefix/suffix K/V).
//
// A denoise step has only block-many queries per head, so the keys are split
// across CTAs (flash-decoding): CTA (split, q-tile, head, seq) streams its key
// range through a two-stage TMA ring (3-D tensor map over the cache, 128-byte
// swizzle), computes S = Q K^T and O = P V on the tensor cores
// (mma.sync m16n8k16 bf16 -> f32; the products are small, the K/V bytes are
// what bound the kernel), keeps an online softmax (running max and sum, base-2
// exponentials), merges the warps' key halves through shared memory and the
// key splits through a workspace: the last split to finish combines all
// partials in split order.
//
// Split precision (kv_lo = 1): q, K and V each come as a bf16 pair x = hi + lo
// (lo = bf16(x - hi), about 16 significant bits together), and so does P in
// registers; S = Qh Kh + Ql Kh + Qh Kl and O = Ph Vh + Pl Vh + Ph Vl (the lo*lo
// terms are below 2^-16 relative).  With bf16 alone the rounding of the
// cached K/V moves final hidden states by a few 1e-3 relative.
#pragma once

#include <climits>

#include "ptx.cuh"

namespace dllm {

struct AttnParams {
  const uint16_t* q;   // [b*R][H][HD]
  const uint16_t* q_lo;  // low halves of q (kv_lo = 1), else unused
  uint16_t* o;         // [b*R][H*HD]
  uint16_t* o_lo;      // low halves (o - bf16(o)), or null
  int R, b, H, T;      // query rows per sequence, sequences, heads, valid keys
  int z_k0, z_v0;      // plane of (seq 0, head 0) in the K and V maps; plane = z0 + seq*H + head
  int z_kl0, z_vl0;    // the same for the low halves of K and V (kv_lo = 1)
  int kv_lo;           // 1: split-precision q, K, V and P
  // block-causal mask (mask_B > 0): the query at position p = row0 + row sees
  // keys below p's block end: mask_P for prompt positions (p < mask_P), else
  // mask_P + ((p - mask_P) / mask_B + 1) * mask_B.  mask_B = 0: every key.
  int row0, mask_P, mask_B;
  int q_tiles, splits, kps;  // query tiles per (seq, head), key splits, keys per split (multiple of 64)
  int n_whole;         // tensor-core kernel: leading query tiles run unsplit, the rest in `splits` splits
  float scale_log2;    // log2(e) / sqrt(HD)
  float* ws_o;         // [works][splits][QT][HD]
  float* ws_ml;        // [works][splits][QT][2]
  int* counters;       // [works]
  int* err;
};

// LO: room for the low halves of K and V (split precision); without them a
// 32-key CTA needs 50 KB instead of 83 KB and four fit on an SM instead of two.
template <int HD, int KT, bool LO = true>
struct AttnCfg {
  static constexpr int TILE_BYTES = KT * HD * 2;     // one of K, V, K lo, V lo
  static constexpr int STAGES = 2;
  static constexpr int PARTS = (KT == 32 && LO) ? 2 : 1;   // 32-key tiles leave room for the low halves
  static constexpr int SMEM_BYTES = 1024 + STAGES * 2 * PARTS * TILE_BYTES + 32 * HD * 4 + 32 * 2 * 4 + 64;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// The bf16 residuals of a pair against its packed bf16 values hv.
__device__ __forceinline__ uint32_t pack_lo(float a, float b, uint32_t hv) {
  return pack_bf16(a - __uint_as_float(hv << 16), b - __uint_as_float(hv & 0xffff0000u));
}

// Store a pair of outputs as bf16 and, when o_lo is set, their bf16 residuals.
__device__ __forceinline__ void store_pair(uint16_t* o, uint16_t* o_lo, long long idx, float a, float b) {
  const uint32_t hv = pack_bf16(a, b);
  *reinterpret_cast<uint32_t*>(&o[idx]) = hv;
  if (o_lo) {
    const float ah = __uint_as_float(hv << 16), bh = __uint_as_float(hv & 0xffff0000u);
    *reinterpret_cast<uint32_t*>(&o_lo[idx]) = pack_bf16(a - ah, b - bh);
  }
}

// Byte offset of the 16-byte chunk `ch` (8 bf16 along the head dim) of key row
// `r` in a TMA 128B-swizzled tile stored as HD/64 boxes of [KT keys][128 B].
template <int KT>
__device__ __forceinline__ uint32_t swz_off(int r, int ch) {
  return (uint32_t)((ch >> 3) * (KT * 128) + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// The last split of a work (seq, head, query tile of QT rows) combines the
// partials (o, m, l) of all splits, in split order: per row, weights
// exp2(m_s - M) / L computed once, then every output element is an
// independent weighted sum over the splits.  128 threads (named barrier 2);
// xo holds at least QT * splits floats.  Returns true.
template <int HD, int QT>
__device__ __forceinline__ bool attn_merge(const AttnParams& p, long long work, int qt, int head, int seq, float* xo,
                                           int tid) {
  const float* base_o = p.ws_o + work * p.splits * QT * HD;
  const float* base_ml = p.ws_ml + work * p.splits * QT * 2;
  float* wn = xo;   // [QT][splits] normalised split weights (the key-group buffer is free now)
  const int S = p.splits;
  // The partials were written by other CTAs: every load is an L2 round trip,
  // so they are issued in unrolled, predicated batches rather than one
  // dependent load per split.
  for (int rl = tid; rl < QT; rl += 128) {
    float M = -INFINITY;
    for (int s0 = 0; s0 < S; s0 += 8) {
      float mv[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mv[t] = s0 + t < S ? __ldcg(&base_ml[((s0 + t) * QT + rl) * 2]) : -INFINITY;
#pragma unroll
      for (int t = 0; t < 8; ++t) M = fmaxf(M, mv[t]);
    }
    const float u = (M == -INFINITY) ? 0.0f : M;
    float L = 0.0f;
    for (int s0 = 0; s0 < S; s0 += 8) {
      float2 ml[8];
#pragma unroll
      for (int t = 0; t < 8; ++t)
        ml[t] = s0 + t < S ? __ldcg(reinterpret_cast<const float2*>(&base_ml[((s0 + t) * QT + rl) * 2]))
                           : make_float2(-INFINITY, 0.0f);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (s0 + t < S) {
          const float a = exp2f(ml[t].x - u);
          wn[rl * S + s0 + t] = a;
          L += ml[t].y * a;
        }
      }
    }
    const float il = L > 0.0f ? 1.0f / L : 0.0f;
    for (int s = 0; s < S; ++s) wn[rl * S + s] *= il;
  }
  named_bar_sync(2, 128);
  // four output vectors per thread and pass, four splits per batch: sixteen
  // loads in flight; the sum over splits keeps split order
  for (int e0 = tid; e0 < QT * HD / 4; e0 += 4 * 128) {
    float4 acc[4];
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) acc[u4] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 4) {
      float4 v[4][4];
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const int e4 = e0 + u4 * 128;
        const int rl = (e4 * 4) / HD, col = e4 * 4 - rl * HD;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          v[u4][t] = (e4 < QT * HD / 4 && s0 + t < S)
                         ? __ldcg(reinterpret_cast<const float4*>(&base_o[((s0 + t) * QT + rl) * HD + col]))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const int e4 = e0 + u4 * 128;
        const int rl = (e4 * 4) / HD;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (e4 < QT * HD / 4 && s0 + t < S) {
            const float w = wn[rl * S + s0 + t];
            acc[u4].x += v[u4][t].x * w;
            acc[u4].y += v[u4][t].y * w;
            acc[u4].z += v[u4][t].z * w;
            acc[u4].w += v[u4][t].w * w;
          }
        }
      }
    }
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) {
      const int e4 = e0 + u4 * 128;
      if (e4 >= QT * HD / 4) continue;
      const int rl = (e4 * 4) / HD, col = e4 * 4 - rl * HD;
      const int row = qt * QT + rl;
      if (row >= p.R) continue;
      const float4 a4 = acc[u4];
      const long long oi = ((long long)seq * p.R + row) * p.H * HD + head * HD + col;
      store_pair(p.o, p.o_lo, oi, a4.x, a4.y);
      store_pair(p.o, p.o_lo, oi + 2, a4.z, a4.w);
    }
  }
  return true;
}

// One work item (key split, query tile, head, sequence) of block attention,
// run by a group of 128 threads (tid 0..127, named barrier 2).  sK/sV hold ST
// stages of [KT keys][HD] tiles (1024-byte aligned), each stage followed by its
// low-half tile when p.kv_lo is set; xo at least 32*HD floats, full[ST]
// mbarriers initialised to count 1.  tcount counts the tiles this group has
// loaded through `full` so far (phase parity across items); it is advanced by
// the item's tile count.  stamps (optional, thread 0): [0] keys done, [1]
// split partial stored and counted.  Returns true when this call wrote the final output
// rows of its (sequence, head, query tile): the only split, or the last split
// to finish, which merges all of them.
template <int HD, int WQ, int ST, int KT>
__device__ __forceinline__ bool attn_item(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                                          int split, int qt, int head, int seq, uint8_t* sK, uint8_t* sV, float* xo,
                                          uint64_t* full, int* bcast, uint32_t& tcount, int tid,
                                          unsigned long long* stamps = nullptr) {
  constexpr int TILE_BYTES = KT * HD * 2;
  constexpr int WK = 4 / WQ;
  constexpr int QT = 16 * WQ;
  constexpr int KW = KT / WK;      // keys per warp per tile
  constexpr int NT = KW / 8;       // n8 tiles of S per warp
  constexpr int KS = HD / 16;      // k16 steps of Q K^T
  constexpr int OT = HD / 8;       // n8 tiles of O
  static_assert(QT <= 64, "query tile");
  float* xml = xo + 32 * HD;       // [32][2]
  const int warp = tid >> 5, lane = tid & 31;
  const int wq = warp % WQ, wk = warp / WQ;
  const int g = lane >> 2, t4 = lane & 3;
  const int k_beg = split * p.kps;
  int k_end = min(p.T, k_beg + p.kps);
  int lim_lo = INT_MAX, lim_hi = INT_MAX;   // key limits of this thread's two query rows
  if (p.mask_B > 0) {
    auto key_limit = [&](int row) {
      const int pos = p.row0 + row;
      return pos < p.mask_P ? p.mask_P : p.mask_P + ((pos - p.mask_P) / p.mask_B + 1) * p.mask_B;
    };
    const int qr = qt * QT + wq * 16 + g;
    lim_lo = key_limit(qr);
    lim_hi = key_limit(qr + 8);
    // limits grow with position: the tile's last row bounds the keys to visit
    k_end = min(k_end, key_limit(min(qt * QT + QT, p.R) - 1));
  }
  const int ntiles = k_end > k_beg ? (k_end - k_beg + KT - 1) / KT : 0;
  const int zk = p.z_k0 + seq * p.H + head, zv = p.z_v0 + seq * p.H + head;
  const int zkl = p.z_kl0 + seq * p.H + head, zvl = p.z_vl0 + seq * p.H + head;
  const bool lo = KT == 32 && p.kv_lo != 0;   // 64-key tiles are bf16 only (no room for the low halves)
  const int stage_bytes = (lo ? 2 : 1) * TILE_BYTES;   // per stage of sK (and of sV): hi tile, then lo tile

  const uint64_t pol = policy_evict_first();
  auto issue = [&](int t, int s) {
    const int key0 = k_beg + t * KT;
    mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * stage_bytes));
#pragma unroll
    for (int bx = 0; bx < HD / 64; ++bx) {
      tma_load_3d(sK + s * stage_bytes + bx * (KT * 128), tmK, &full[s], bx * 64, key0, zk, pol);
      tma_load_3d(sV + s * stage_bytes + bx * (KT * 128), tmV, &full[s], bx * 64, key0, zv, pol);
      if (lo) {
        tma_load_3d(sK + s * stage_bytes + TILE_BYTES + bx * (KT * 128), tmK, &full[s], bx * 64, key0, zkl, pol);
        tma_load_3d(sV + s * stage_bytes + TILE_BYTES + bx * (KT * 128), tmV, &full[s], bx * 64, key0, zvl, pol);
      }
    }
  };
  const uint32_t tc0 = tcount;
  if (tid == 0)
    for (int t = 0; t < ST && t < ntiles; ++t) issue(t, (int)((tc0 + t) % ST));

  // Q fragments of this warp's 16 query rows.  With 32 query rows (WQ == 2)
  // the tile (hi and lo) is staged once in xo, 16-byte chunks XOR-swizzled by
  // row so that ldmatrix reads are conflict-free, and the fragments are
  // re-read per k-step: holding all of them in registers (64 per thread) made
  // the persistent step kernel spill.  xo is free until the key loop ends.
  const int qrow0 = qt * QT + wq * 16;
  uint32_t qa[WQ == 2 ? 1 : KS][4], ql[WQ == 2 ? 1 : KS][4];
  uint16_t* const qs_hi = reinterpret_cast<uint16_t*>(xo);
  uint16_t* const qs_lo = qs_hi + 32 * HD;
  if constexpr (WQ == 2) {
    constexpr int CH = HD / 8;                   // 16-byte chunks per row
    for (int e = tid; e < 32 * CH; e += 128) {
      const int rl = e / CH, c = e - rl * CH;
      const int row = qt * QT + rl;
      uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = hv;
      if (row < p.R) {
        // L2-coherent loads: q was written by other CTAs of the same launch (persistent step)
        const long long base = (((long long)seq * p.R + row) * p.H + head) * HD + c * 8;
        hv = __ldcg(reinterpret_cast<const uint4*>(p.q + base));
        if (lo) lv = __ldcg(reinterpret_cast<const uint4*>(p.q_lo + base));
      }
      const int pc = c ^ (rl & 7);
      *reinterpret_cast<uint4*>(qs_hi + rl * HD + pc * 8) = hv;
      *reinterpret_cast<uint4*>(qs_lo + rl * HD + pc * 8) = lv;
    }
    named_bar_sync(2, 128);
  } else {
    const long long base_lo = (((long long)seq * p.R + qrow0 + g) * p.H + head) * HD;
    const long long base_hi = base_lo + 8LL * p.H * HD;
    const bool lo_ok = qrow0 + g < p.R, hi_ok = qrow0 + g + 8 < p.R;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const uint32_t* ql32 = reinterpret_cast<const uint32_t*>(lo ? p.q_lo : p.q);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int c0 = kk * 16 + 2 * t4;
      // L2-coherent loads: q was written by other CTAs of the same launch (persistent step)
      qa[kk][0] = lo_ok ? __ldcg(&q32[(base_lo + c0) >> 1]) : 0u;
      qa[kk][1] = hi_ok ? __ldcg(&q32[(base_hi + c0) >> 1]) : 0u;
      qa[kk][2] = lo_ok ? __ldcg(&q32[(base_lo + c0 + 8) >> 1]) : 0u;
      qa[kk][3] = hi_ok ? __ldcg(&q32[(base_hi + c0 + 8) >> 1]) : 0u;
      ql[kk][0] = lo && lo_ok ? __ldcg(&ql32[(base_lo + c0) >> 1]) : 0u;
      ql[kk][1] = lo && hi_ok ? __ldcg(&ql32[(base_hi + c0) >> 1]) : 0u;
      ql[kk][2] = lo && lo_ok ? __ldcg(&ql32[(base_lo + c0 + 8) >> 1]) : 0u;
      ql[kk][3] = lo && hi_ok ? __ldcg(&ql32[(base_hi + c0 + 8) >> 1]) : 0u;
    }
  }

  float oacc[OT][4];
#pragma unroll
  for (int i = 0; i < OT; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.0f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.0f, l_hi = 0.0f;
  bool failed = false;

  for (int t = 0; t < ntiles; ++t) {
    const uint32_t tg = tc0 + t;
    const int s = (int)(tg % ST);
    if (!failed && !mbar_wait(&full[s], (tg / ST) & 1u, nullptr, p.err, ERR_ATTN_FULL))
      failed = true;
    if (!failed) {
      const uint32_t kb = smem_u32(sK + s * stage_bytes);
      const uint32_t vb = smem_u32(sV + s * stage_bytes);
      const int key_w = wk * KW;       // first key of this warp inside the tile
      // S = Q K^T.  Six independent accumulators per n8 tile (the hi*hi,
      // lo*hi and hi*lo products, each split over even and odd k16 steps)
      // keep the dependent MMA chains short; they are summed in a fixed order.
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float acc[6][4];
#pragma unroll
        for (int u = 0; u < 6; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.0f;
        const int r = key_w + nt * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < KS; kk += 2) {
          const int ch = 2 * kk + (lane >> 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz_off<KT>(r, ch), b0, b1, b2, b3);
          uint32_t fa0[4], fa1[4], fl0[4], fl1[4];
          if constexpr (WQ == 2) {
            // rows wq*16 + 0..15: lanes 8-15 and 24-31 address rows 8-15,
            // lanes 16-31 the second 8 dims of the k-step
            const int rr = wq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int c0 = (2 * kk + (lane >> 4)) ^ (rr & 7), c1 = (2 * kk + 2 + (lane >> 4)) ^ (rr & 7);
            ldsm_x4(smem_u32(qs_hi + rr * HD + c0 * 8), fa0[0], fa0[1], fa0[2], fa0[3]);
            ldsm_x4(smem_u32(qs_hi + rr * HD + c1 * 8), fa1[0], fa1[1], fa1[2], fa1[3]);
            if (lo) {
              ldsm_x4(smem_u32(qs_lo + rr * HD + c0 * 8), fl0[0], fl0[1], fl0[2], fl0[3]);
              ldsm_x4(smem_u32(qs_lo + rr * HD + c1 * 8), fl1[0], fl1[1], fl1[2], fl1[3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              fa0[i] = qa[kk][i];
              fa1[i] = qa[kk + 1][i];
              fl0[i] = ql[kk][i];
              fl1[i] = ql[kk + 1][i];
            }
          }
          mma16816(acc[0], fa0, b0, b1);
          mma16816(acc[1], fa1, b2, b3);
          if (lo) {
            mma16816(acc[2], fl0, b0, b1);
            mma16816(acc[3], fl1, b2, b3);
            ldsm_x4(kb + TILE_BYTES + swz_off<KT>(r, ch), b0, b1, b2, b3);
            mma16816(acc[4], fa0, b0, b1);
            mma16816(acc[5], fa1, b2, b3);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sacc[nt][e] = lo ? ((acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e])) + (acc[4][e] + acc[5][e])
                           : acc[0][e] + acc[1][e];
      }
      // online softmax (base 2)
      const int key_base = k_beg + t * KT + key_w;
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_base + nt * 8 + 2 * t4 + e;
          const bool ok_lo = key < k_end && key < lim_lo, ok_hi = key < k_end && key < lim_hi;
          sacc[nt][e] = ok_lo ? sacc[nt][e] * p.scale_log2 : -INFINITY;
          sacc[nt][2 + e] = ok_hi ? sacc[nt][2 + e] * p.scale_log2 : -INFINITY;
          mx_lo = fmaxf(mx_lo, sacc[nt][e]);
          mx_hi = fmaxf(mx_hi, sacc[nt][2 + e]);
        }
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      // The reference max of a row only moves when a tile's max exceeds it by
      // more than 8 (a factor 2^8 in probability); otherwise P = exp2(s - m)
      // <= 256, and O and l keep their scale: the same sums, referred to a
      // slightly smaller max, with the rescale of O skipped in most tiles.
      const bool up_lo = mx_lo > m_lo + 8.0f, up_hi = mx_hi > m_hi + 8.0f;
      const float mn_lo = up_lo ? mx_lo : m_lo, mn_hi = up_hi ? mx_hi : m_hi;
      const float use_lo = (mn_lo == -INFINITY) ? 0.0f : mn_lo;
      const float use_hi = (mn_hi == -INFINITY) ? 0.0f : mn_hi;
      const float corr_lo = up_lo ? exp2f(m_lo - use_lo) : 1.0f, corr_hi = up_hi ? exp2f(m_hi - use_hi) : 1.0f;
      m_lo = mn_lo;
      m_hi = mn_hi;
      float sum_lo = 0.0f, sum_hi = 0.0f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sacc[nt][0] = exp2f(sacc[nt][0] - use_lo);
        sacc[nt][1] = exp2f(sacc[nt][1] - use_lo);
        sacc[nt][2] = exp2f(sacc[nt][2] - use_hi);
        sacc[nt][3] = exp2f(sacc[nt][3] - use_hi);
        sum_lo += sacc[nt][0] + sacc[nt][1];
        sum_hi += sacc[nt][2] + sacc[nt][3];
      }
      sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 1);
      sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 2);
      sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 1);
      sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 2);
      l_lo = l_lo * corr_lo + sum_lo;
      l_hi = l_hi * corr_hi + sum_hi;
      if (up_lo || up_hi) {
#pragma unroll
        for (int i = 0; i < OT; ++i) {
          oacc[i][0] *= corr_lo;
          oacc[i][1] *= corr_lo;
          oacc[i][2] *= corr_hi;
          oacc[i][3] *= corr_hi;
        }
      }
      // O += P V
#pragma unroll
      for (int j = 0; j < KW / 16; ++j) {
        uint32_t pa[4], pl[4];
        pa[0] = pack_bf16(sacc[2 * j][0], sacc[2 * j][1]);
        pa[1] = pack_bf16(sacc[2 * j][2], sacc[2 * j][3]);
        pa[2] = pack_bf16(sacc[2 * j + 1][0], sacc[2 * j + 1][1]);
        pa[3] = pack_bf16(sacc[2 * j + 1][2], sacc[2 * j + 1][3]);
        if (lo) {
          pl[0] = pack_lo(sacc[2 * j][0], sacc[2 * j][1], pa[0]);
          pl[1] = pack_lo(sacc[2 * j][2], sacc[2 * j][3], pa[1]);
          pl[2] = pack_lo(sacc[2 * j + 1][0], sacc[2 * j + 1][1], pa[2]);
          pl[3] = pack_lo(sacc[2 * j + 1][2], sacc[2 * j + 1][3], pa[3]);
        }
        const int mi = lane >> 3;
        const int r = key_w + j * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ot = 0; ot < OT; ot += 2) {
          const int ch = ot + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz_off<KT>(r, ch), b0, b1, b2, b3);
          mma16816(oacc[ot], pa, b0, b1);
          mma16816(oacc[ot + 1], pa, b2, b3);
          if (lo) {
            mma16816(oacc[ot], pl, b0, b1);
            mma16816(oacc[ot + 1], pl, b2, b3);
            ldsm_x4_t(vb + TILE_BYTES + swz_off<KT>(r, ch), b0, b1, b2, b3);
            mma16816(oacc[ot], pa, b0, b1);
            mma16816(oacc[ot + 1], pa, b2, b3);
          }
        }
      }
    }
    named_bar_sync(2, 128);
    if (tid == 0 && !failed && t + ST < ntiles) issue(t + ST, s);
  }
  tcount = tc0 + ntiles;
  if (stamps && tid == 0) stamps[0] = globaltimer();   // keys done

  // combine the key groups of a CTA (WK == 2): group 1 hands its state to group 0
  if constexpr (WK == 2) {
    if (wk == 1) {
      const int rl = wq * 16 + g;
#pragma unroll
      for (int i = 0; i < OT; ++i) {
        const int col = i * 8 + 2 * t4;
        xo[rl * HD + col] = oacc[i][0];
        xo[rl * HD + col + 1] = oacc[i][1];
        xo[(rl + 8) * HD + col] = oacc[i][2];
        xo[(rl + 8) * HD + col + 1] = oacc[i][3];
      }
      if (t4 == 0) {
        xml[rl * 2] = m_lo;
        xml[rl * 2 + 1] = l_lo;
        xml[(rl + 8) * 2] = m_hi;
        xml[(rl + 8) * 2 + 1] = l_hi;
      }
    }
    named_bar_sync(2, 128);
    if (wk == 0) {
      const int rl = wq * 16 + g;
      const float m1_lo = xml[rl * 2], l1_lo = xml[rl * 2 + 1];
      const float m1_hi = xml[(rl + 8) * 2], l1_hi = xml[(rl + 8) * 2 + 1];
      const float M_lo = fmaxf(m_lo, m1_lo), M_hi = fmaxf(m_hi, m1_hi);
      const float u_lo = (M_lo == -INFINITY) ? 0.0f : M_lo, u_hi = (M_hi == -INFINITY) ? 0.0f : M_hi;
      const float a0_lo = exp2f(m_lo - u_lo), a1_lo = exp2f(m1_lo - u_lo);
      const float a0_hi = exp2f(m_hi - u_hi), a1_hi = exp2f(m1_hi - u_hi);
#pragma unroll
      for (int i = 0; i < OT; ++i) {
        const int col = i * 8 + 2 * t4;
        oacc[i][0] = oacc[i][0] * a0_lo + xo[rl * HD + col] * a1_lo;
        oacc[i][1] = oacc[i][1] * a0_lo + xo[rl * HD + col + 1] * a1_lo;
        oacc[i][2] = oacc[i][2] * a0_hi + xo[(rl + 8) * HD + col] * a1_hi;
        oacc[i][3] = oacc[i][3] * a0_hi + xo[(rl + 8) * HD + col + 1] * a1_hi;
      }
      l_lo = l_lo * a0_lo + l1_lo * a1_lo;
      l_hi = l_hi * a0_hi + l1_hi * a1_hi;
      m_lo = M_lo;
      m_hi = M_hi;
    }
  }

  const bool writer = (wk == 0);
  const int row_lo = qrow0 + g, row_hi = qrow0 + g + 8;
  if (p.splits == 1) {
    if (writer) {
      const float il = l_lo > 0.0f ? 1.0f / l_lo : 0.0f, ih = l_hi > 0.0f ? 1.0f / l_hi : 0.0f;
#pragma unroll
      for (int i = 0; i < OT; ++i) {
        const int col = i * 8 + 2 * t4;
        if (row_lo < p.R)
          store_pair(p.o, p.o_lo, ((long long)seq * p.R + row_lo) * p.H * HD + head * HD + col, oacc[i][0] * il,
                     oacc[i][1] * il);
        if (row_hi < p.R)
          store_pair(p.o, p.o_lo, ((long long)seq * p.R + row_hi) * p.H * HD + head * HD + col, oacc[i][2] * ih,
                     oacc[i][3] * ih);
      }
    }
    return true;
  }

  const long long work = ((long long)seq * p.H + head) * p.q_tiles + qt;
  const long long wbase = work * p.splits + split;
  if (writer) {
    float* wo = p.ws_o + wbase * QT * HD;
    float* wml = p.ws_ml + wbase * QT * 2;
    const int rl = wq * 16 + g;
#pragma unroll
    for (int i = 0; i < OT; ++i) {
      const int col = i * 8 + 2 * t4;
      __stcg(reinterpret_cast<float2*>(&wo[rl * HD + col]), make_float2(oacc[i][0], oacc[i][1]));
      __stcg(reinterpret_cast<float2*>(&wo[(rl + 8) * HD + col]), make_float2(oacc[i][2], oacc[i][3]));
    }
    if (t4 == 0) {
      __stcg(reinterpret_cast<float2*>(&wml[rl * 2]), make_float2(m_lo, l_lo));
      __stcg(reinterpret_cast<float2*>(&wml[(rl + 8) * 2]), make_float2(m_hi, l_hi));
    }
  }
  // the barrier orders every thread's partial stores before thread 0's
  // release; its acquire plus the next barrier order the reads after
  named_bar_sync(2, 128);
  if (tid == 0) {
    const int old = atomic_add_acq_rel_gpu(&p.counters[work], 1);
    const int last = (old == p.splits - 1);
    if (last) p.counters[work] = 0;
    *bcast = last;
    if (stamps) stamps[1] = globaltimer();               // partial stored and counted
  }
  named_bar_sync(2, 128);
  if (!*bcast) return false;
  return attn_merge<HD, QT>(p, work, qt, head, seq, xo, tid);
}

// Standalone launch: one work item per CTA.  KT = 32 also takes the low
// halves (kv_lo); KT = 64 is bf16 only.
template <int HD, int WQ, int KT, bool LO = true>
__global__ void __launch_bounds__(128) attn_kernel(const __grid_constant__ CUtensorMap tmK,
                                                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = AttnCfg<HD, KT, LO>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::STAGES * C::PARTS * C::TILE_BYTES;
  float* xo = reinterpret_cast<float*>(sV + C::STAGES * C::PARTS * C::TILE_BYTES);   // [32][HD] + [32][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(xo + 32 * HD + 64);
  int* bcast = reinterpret_cast<int*>(full + C::STAGES);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();
  griddep_launch_dependents();
  griddep_wait();
  uint32_t tcount = 0;
  attn_item<HD, WQ, C::STAGES, KT>(&tmK, &tmV, p, blockIdx.x, blockIdx.y % p.q_tiles, blockIdx.y / p.q_tiles,
                               blockIdx.z, sK, sV, xo, full, bcast, tcount, threadIdx.x);
}

}  // namespace dllm
