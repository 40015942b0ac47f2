// Non-causal attention on the tensor cores for long query sets (the refresh's
// full forward, PrefixCache and no-cache steps): eq. 3 of the zhongzhuzhou.org
// notes, section 2, with every query of a 128-row tile reading every key of
// its sequence (or, under the block-causal mask, the keys below its block's
// end).
//
// One CTA per (128-query tile, key split, head, sequence) walks its keys in
// 64-key tiles (with one split, all keys of the sequence):
//   warp 0     TMA: the query tile once, then K and V tiles (with their low
//              halves in split precision) through a two-stage ring whose K
//              and V halves are refilled separately: a stage's keys as soon
//              as its S product is done, its values once P V is done;
//   warp 1     one thread issues tcgen05.mma: S = Q K^T into one of two
//              64-column TMEM buffers, and O += P V into a HD-column TMEM
//              accumulator with P read from tensor memory; V is read as an
//              MN-major operand straight from the TMA tile (keys along K,
//              head dims along N);
//   warps 2-5  one query row per thread: read S from TMEM, online softmax in
//              base 2 (the row's reference max moves only when a tile's max
//              exceeds it by more than 8, so P <= 256 and O is rescaled
//              rarely, in TMEM), write P as bf16 (hi and lo) into one of two
//              TMEM buffers (the row's lane, keys packed two per column), and
//              at the end O / l to global memory.
// S of tile t+1 runs on the tensor cores while the softmax of tile t runs,
// and the softmax of tile t+1 writes its P while P V of tile t runs.
// With several key splits each CTA stores its partial (O, m, l) and the last
// split of a query tile to finish merges them (the key-split kernel's merge,
// 128 rows); splits are planned when there are too few query tiles to fill
// the GPU evenly.
//
// Split precision (kv_lo = 1): q, K, V and P are bf16 pairs x = hi + lo;
// S = Qh Kh + Ql Kh + Qh Kl and O += Ph Vh + Pl Vh + Ph Vl (lo*lo dropped).
#pragma once

#include <climits>

#include "attention.cuh"
#include "ptx.cuh"

namespace dllm {

template <int HD>
struct AttnTcCfg {
  static constexpr int KT = 64;                      // keys per tile
  static constexpr int Q_BYTES = 128 * HD * 2;       // one part (hi or lo) of the query tile
  static constexpr int KV_BYTES = KT * HD * 2;       // one part of a K or V tile
  static constexpr int STAGE_BYTES = 4 * KV_BYTES;   // K hi, K lo, V hi, V lo
  static constexpr int MERGE_BYTES = 128 * 8 * 4;    // split merge weights: 128 rows x up to 8 splits
  static constexpr int SMEM_BYTES = 1024 + 2 * Q_BYTES + 2 * STAGE_BYTES + MERGE_BYTES + 256;
  static constexpr int S_COL = 0;                    // two S buffers of KT columns
  static constexpr int O_COL = 2 * KT;               // O accumulator, HD columns
  static constexpr int P_COL = 2 * KT + HD;          // two P buffers of KT columns: KT/2 hi, KT/2 lo
  static constexpr int TMEM_COLS = 512;
  static_assert(P_COL + 2 * KT <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Shared-memory descriptor of an MN-major operand written by TMA with the
// 128-byte swizzle: each 128-byte row holds 64 consecutive MN elements of one
// K index, 8 K rows form a 1024-byte atom (SBO between atoms along K), and
// the next 64 MN elements start lbo bytes further.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// 32 lanes x 32 consecutive 32-bit columns written back from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Key limit of query position pos: T, or under the block-causal mask the end
// of pos's block (the prompt counts as one block).
__device__ __forceinline__ int tc_key_limit(const AttnParams& p, int pos) {
  if (p.mask_B <= 0) return p.T;
  const int lim = pos < p.mask_P ? p.mask_P : p.mask_P + ((pos - p.mask_P) / p.mask_B + 1) * p.mask_B;
  return lim < p.T ? lim : p.T;
}

// 1-D grid, 192 threads.  Query tiles (items, numbered (seq * H + head) *
// q_tiles + qt, so that neighbouring CTAs share a head's keys in L2): the
// first p.n_whole run unsplit, one CTA each; every later one in p.splits key
// ranges of p.kps keys (a multiple of 64), merged in the workspace (p.ws_o,
// p.ws_ml, p.counters, indexed from the first split item).  Grid:
// n_whole + (items - n_whole) * splits CTAs.  tmQ/tmQlo: 2-D maps over
// q / q_lo [b*R][H*HD] with 128-row boxes; tmK/tmV: 3-D maps over the K and V
// planes with 64-key boxes (the same map may serve both).
template <int HD>
__global__ void __launch_bounds__(192, 1) attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                        const __grid_constant__ CUtensorMap tmQlo,
                                                        const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = AttnTcCfg<HD>;
  constexpr int KT = C::KT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // Q hi, Q lo
  uint8_t* sKV = sQ + 2 * C::Q_BYTES;                   // per stage: K hi, K lo, V hi, V lo
  float* s_merge = reinterpret_cast<float*>(sKV + 2 * C::STAGE_BYTES);   // split merge weights
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + 2 * C::STAGE_BYTES + C::MERGE_BYTES);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;     // [2] a stage's K (and K lo) landed
  uint64_t* kempty = bars + 3;    // [2] its S product is done with it
  uint64_t* sfull = bars + 5;     // [2]
  uint64_t* sfree = bars + 7;     // [2]
  uint64_t* pready = bars + 9;    // [2] a P buffer written by the four softmax warps
  uint64_t* pvdone = bars + 11;   // [2] P V of the tile in a P buffer done
  uint64_t* vfull = bars + 13;    // [2] a stage's V (and V lo) landed
  uint64_t* vempty = bars + 15;   // [2] its P V product is done with it
  uint64_t* mdone = bars + 17;    // every MMA of the CTA finished (before TMEM is freed)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bcast = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int item, split, splits;
  if ((int)blockIdx.x < p.n_whole) {
    item = (int)blockIdx.x;
    split = 0;
    splits = 1;
  } else {
    const int r = (int)blockIdx.x - p.n_whole;
    splits = p.splits > 1 ? p.splits : 1;
    item = p.n_whole + r / splits;
    split = r - (r / splits) * splits;
  }
  const int qt = item % p.q_tiles, head = (item / p.q_tiles) % p.H, seq = item / (p.q_tiles * p.H);
  const bool lo = p.kv_lo != 0;
  const int parts = lo ? 2 : 1;
  // keys this tile's rows see at most: limits grow with the position
  const int last_row = min(p.R, qt * 128 + 128) - 1;
  const int k_lim = tc_key_limit(p, p.row0 + last_row);
  // this split's keys [k_beg, k_stop), tiles t0 .. t0 + nt - 1
  const int k_beg = splits > 1 ? split * p.kps : 0;
  const int k_stop = splits > 1 ? min(k_lim, k_beg + p.kps) : k_lim;
  const int nt = k_stop > k_beg ? (k_stop - k_beg + KT - 1) / KT : 0;
  const int t0 = k_beg / KT;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
      mbar_init(&sfull[s], 1);
      mbar_init(&sfree[s], 4);
      mbar_init(&pready[s], 4);
      mbar_init(&pvdone[s], 1);
    }
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();   // the other query tiles of this head read the same keys
      const int row = seq * p.R + qt * 128;
      mbar_arrive_expect_tx(qfull, (uint32_t)(parts * C::Q_BYTES));
      for (int part = 0; part < parts; ++part)
        for (int bx = 0; bx < HD / 64; ++bx)
          tma_load_2d(sQ + part * C::Q_BYTES + bx * (128 * 128), part ? &tmQlo : &tmQ, qfull, head * HD + bx * 64,
                      row, pol_q);
      const int zk = p.z_k0 + seq * p.H + head, zv = p.z_v0 + seq * p.H + head;
      const int zkl = p.z_kl0 + seq * p.H + head, zvl = p.z_vl0 + seq * p.H + head;
      // K of tile t waits for S of tile t-2, V of tile t for P V of tile
      // t-2; since S runs about a tile ahead of P V, keys are requested a
      // tile earlier than a whole-stage refill would allow
      int k_issued = 0, v_issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int s = t & 1;
        uint8_t* st = sKV + s * C::STAGE_BYTES;
        if (t >= 2 && !mbar_wait(&kempty[s], (uint32_t)((t >> 1) - 1) & 1u, abort_flag, p.err, ERR_ATTN_FULL)) break;
        mbar_arrive_expect_tx(&kfull[s], (uint32_t)(parts * C::KV_BYTES));
        for (int bx = 0; bx < HD / 64; ++bx) {
          tma_load_3d(st + 0 * C::KV_BYTES + bx * (KT * 128), &tmK, &kfull[s], bx * 64, (t0 + t) * KT, zk, pol_kv);
          if (lo)
            tma_load_3d(st + 1 * C::KV_BYTES + bx * (KT * 128), &tmK, &kfull[s], bx * 64, (t0 + t) * KT, zkl, pol_kv);
        }
        k_issued = t + 1;
        if (t >= 2 && !mbar_wait(&vempty[s], (uint32_t)((t >> 1) - 1) & 1u, abort_flag, p.err, ERR_ATTN_FULL)) break;
        mbar_arrive_expect_tx(&vfull[s], (uint32_t)(parts * C::KV_BYTES));
        for (int bx = 0; bx < HD / 64; ++bx) {
          tma_load_3d(st + 2 * C::KV_BYTES + bx * (KT * 128), &tmV, &vfull[s], bx * 64, (t0 + t) * KT, zv, pol_kv);
          if (lo)
            tma_load_3d(st + 3 * C::KV_BYTES + bx * (KT * 128), &tmV, &vfull[s], bx * 64, (t0 + t) * KT, zvl, pol_kv);
        }
        v_issued = t + 1;
      }
      // nothing may land in shared memory after the CTA is gone
      mbar_wait(qfull, 0u, nullptr, p.err, ERR_ATTN_FULL);
      for (int t = k_issued - 2 < 0 ? 0 : k_issued - 2; t < k_issued; ++t)
        mbar_wait(&kfull[t & 1], (uint32_t)(t >> 1) & 1u, nullptr, p.err, ERR_ATTN_FULL);
      for (int t = v_issued - 2 < 0 ? 0 : v_issued - 2; t < v_issued; ++t)
        mbar_wait(&vfull[t & 1], (uint32_t)(t >> 1) & 1u, nullptr, p.err, ERR_ATTN_FULL);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, KT);
      const uint32_t idesc_o = idesc_bf16_f32(128, HD) | (1u << 16);   // B (V) MN-major
      const uint32_t q0 = smem_u32(sQ);
      bool ok = mbar_wait(qfull, 0u, abort_flag, p.err, ERR_ATTN_FULL);
      auto issue_s = [&](int t) {
        const int s = t & 1;
        const uint32_t k0 = smem_u32(sKV + s * C::STAGE_BYTES);
        const uint32_t d = tmem + (uint32_t)(C::S_COL + s * KT);
        // (Q part, K part): hi*hi, then lo*hi and hi*lo in split precision
        for (int pr = 0; pr < (lo ? 3 : 1); ++pr) {
          const uint32_t qa = q0 + (pr == 1 ? C::Q_BYTES : 0);
          const uint32_t kb = k0 + (pr == 2 ? C::KV_BYTES : 0);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t bx = kk >> 2, ko = (kk & 3) * 32;
            mma_bf16_ss(d, sdesc_sw128(qa + bx * (128 * 128) + ko), sdesc_sw128(kb + bx * (KT * 128) + ko), idesc_s,
                        (pr > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&sfull[s]);
        mma_commit(&kempty[s]);    // the stage's keys may be refilled
      };
      auto issue_pv = [&](int t) {
        const int s = t & 1;
        const uint32_t v0 = smem_u32(sKV + s * C::STAGE_BYTES + 2 * C::KV_BYTES);
        const uint32_t d = tmem + (uint32_t)C::O_COL;
        const uint32_t pt = tmem + (uint32_t)(C::P_COL + s * KT);   // P hi columns, then P lo
        // (P part, V part): hi*hi, then lo*hi and hi*lo
        for (int pr = 0; pr < (lo ? 3 : 1); ++pr) {
          const uint32_t pa = pt + (pr == 1 ? (uint32_t)(KT / 2) : 0u);
          const uint32_t vb = v0 + (pr == 2 ? C::KV_BYTES : 0);
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            mma_bf16_ts(d, pa + (uint32_t)(kk * 8), sdesc_sw128_mn(vb + kk * 2048, KT * 128), idesc_o,
                        (t > 0 || pr > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&vempty[s]);    // the stage's values may be refilled
        mma_commit(&pvdone[s]);    // the P buffer may be rewritten
      };
      // Issue whichever is ready: P V of the oldest tile whose P is written
      // (it frees a K/V stage for the next load), or S of the next tile once
      // its keys have landed and its S buffer has been read.  Neither waits
      // behind the other.
      int ns = 0, np = 0;
      unsigned long long idle_since = 0;
      uint32_t spins = 0;
      while (ok && np < nt) {
        bool did = false;
        if (np < ns && mbar_test_wait(smem_u32(&pready[np & 1]), (uint32_t)(np >> 1) & 1u) &&
            mbar_test_wait(smem_u32(&vfull[np & 1]), (uint32_t)(np >> 1) & 1u)) {
          tc_fence_after();
          issue_pv(np++);
          did = true;
        }
        if (ns < nt && mbar_test_wait(smem_u32(&kfull[ns & 1]), (uint32_t)(ns >> 1) & 1u) &&
            (ns < 2 || mbar_test_wait(smem_u32(&sfree[ns & 1]), (uint32_t)((ns >> 1) - 1) & 1u))) {
          tc_fence_after();
          issue_s(ns++);
          did = true;
        }
        if (did) {
          idle_since = 0;
          spins = 0;
        } else if ((++spins & 63u) == 0) {
          const unsigned long long now = globaltimer();
          if (idle_since == 0) {
            idle_since = now;
          } else if (*abort_flag || now - idle_since > kWaitLimitNs) {
            if (!*abort_flag) record_error(p.err, ERR_ATTN_FULL);
            *abort_flag = 1;
            ok = false;
          }
        }
      }
      mma_commit(mdone);
      mbar_wait(mdone, 0u, nullptr, p.err, ERR_ATTN_FULL);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int qi = qt * 128 + row;
    const bool valid = qi < p.R;
    const int lim = valid ? tc_key_limit(p, p.row0 + qi) : 0;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      // waits decided warp-wide: the TMEM loads and stores below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[s], (uint32_t)(t >> 1) & 1u, abort_flag, p.err, ERR_ATTN_FULL))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[KT];
      tmem_ld32(trow + (uint32_t)(C::S_COL + s * KT), sv);
      tmem_ld32(trow + (uint32_t)(C::S_COL + s * KT + 32), sv + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[s]);
      const int key0 = k_beg + t * KT;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < KT; ++c) {
        sv[c] = key0 + c < lim ? sv[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, sv[c]);
      }
      const bool up = mx > m + 8.0f;
      const float mn = up ? mx : m;
      const float use = mn == -INFINITY ? 0.0f : mn;
      const float corr = up ? exp2f(m - use) : 1.0f;
      float sum = 0.0f;
#pragma unroll
      for (int c = 0; c < KT; ++c) {
        sv[c] = exp2f(sv[c] - use);
        sum += sv[c];
      }
      l = l * corr + sum;
      m = mn;
      // P buffer s is free once P V of tile t-2 is done; O takes a rescale
      // only after P V of tile t-1
      if (t >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&pvdone[s], (uint32_t)((t >> 1) - 1) & 1u, abort_flag, p.err, ERR_ATTN_FULL))) {
        ok = false;
        break;
      }
      if (t > 0 && __any_sync(0xffffffffu, up)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pvdone[(t - 1) & 1], (uint32_t)((t - 1) >> 1) & 1u, abort_flag, p.err,
                                               ERR_ATTN_FULL))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < HD; c0 += 32) {
          float o[32];
          tmem_ld32(trow + (uint32_t)(C::O_COL + c0), o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(trow + (uint32_t)(C::O_COL + c0), o);
        }
      }
      tc_fence_after();
      // P row into P buffer s: keys 2c and 2c+1 in column c (hi), KT/2 + c (lo)
      {
        float ph[KT / 2], pl[KT / 2];
#pragma unroll
        for (int c = 0; c < KT / 2; ++c) {
          const uint32_t h = pack_bf16(sv[2 * c], sv[2 * c + 1]);
          ph[c] = __uint_as_float(h);
          pl[c] = __uint_as_float(pack_lo(sv[2 * c], sv[2 * c + 1], h));
        }
        const uint32_t pcol = trow + (uint32_t)(C::P_COL + s * KT);
        tmem_st32(pcol, ph);
        if (lo) tmem_st32(pcol + (uint32_t)(KT / 2), pl);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[s]);
    }
    if (ok && nt > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&pvdone[(nt - 1) & 1], (uint32_t)((nt - 1) >> 1) & 1u, abort_flag, p.err,
                                             ERR_ATTN_FULL));
    tc_fence_after();
    if (splits > 1) {
      // this split's partial: O relative to its reference max m, and (m, l)
      const long long work = item - p.n_whole;   // merge slot of this split item
      const long long wrow = (work * splits + split) * 128 + row;
      float* wo = p.ws_o + wrow * HD;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        float o[32];
        if (nt > 0) {
          tmem_ld32(trow + (uint32_t)(C::O_COL + c0), o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          __stcg(reinterpret_cast<float4*>(wo + c0 + 4 * j), make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]));
      }
      __stcg(reinterpret_cast<float2*>(p.ws_ml + wrow * 2), ok ? make_float2(m, l) : make_float2(-INFINITY, 0.0f));
      // the barrier orders every row's stores before the release; the
      // acquire plus the next barrier order the merge's reads after
      named_bar_sync(2, 128);
      if (row == 0) {
        const int old = atomic_add_acq_rel_gpu(&p.counters[work], 1);
        const int last = (old == splits - 1);
        if (last) p.counters[work] = 0;
        *bcast = last;
      }
      named_bar_sync(2, 128);
      if (*bcast) attn_merge<HD, 128>(p, work, qt, head, seq, s_merge, row);
    } else {
      // O / l as bf16 (and its low half)
      const float il = (ok && l > 0.0f) ? 1.0f / l : 0.0f;
      const long long obase = ((long long)seq * p.R + qi) * p.H * HD + head * HD;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        float o[32];
        if (nt > 0) {
          tmem_ld32(trow + (uint32_t)(C::O_COL + c0), o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.0f;
        }
        if (valid) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t h[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = o[8 * j + 2 * e] * il, b = o[8 * j + 2 * e + 1] * il;
              h[e] = pack_bf16(a, b);
              lw[e] = pack_lo(a, b, h[e]);
            }
            *reinterpret_cast<uint4*>(&p.o[obase + c0 + 8 * j]) = make_uint4(h[0], h[1], h[2], h[3]);
            if (p.o_lo)
              *reinterpret_cast<uint4*>(&p.o_lo[obase + c0 + 8 * j]) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
    }
  }
  // Lanes 1-31 of the producer and MMA warps skipped their roles and arrive
  // here first: reconverge each warp before the CTA-wide barrier (an aligned
  // barrier reached by part of a warp would let the warp count as arrived
  // while lane 0 still works, and tensor memory could be freed under the
  // epilogue warps' last reads).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace dllm
