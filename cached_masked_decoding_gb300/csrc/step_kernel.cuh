// Persistent DualCache denoise step: one cooperative launch, one CTA per SM,
// runs every phase of a step - embedding, per layer [QKV+RoPE+K/V write,
// block attention, O-proj+residual+norm, gate/up+SwiGLU, down+residual+norm],
// LM head + softmax statistics, statistic merge + select/commit - separated by
// grid barriers (a global arrival counter, waits bounded in time).
//
// Why: a DualCache step streams ~15 GB of weights through 160 GEMM phases of
// 5-30 us each.  As separate launches every phase pays a pipeline fill (the
// first TMA tile lands ~3 us after the CTA starts) and an epilogue tail.  Here
// the TMA producer walks straight from one GEMM phase into the next: it keeps
// loading the next phase's weight tiles into the shared-memory ring (weights
// depend on nothing) while the other CTAs finish the current phase's
// epilogues, and only the activation tiles wait for the barrier.
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 tcgen05.mma issuer,
// warps 2-5 "workers": GEMM epilogues, and the embedding, attention and merge
// phases.  The ring, the TMEM double buffer and the attention mbarriers keep
// their phase parity across phases through running counters.
#pragma once

#include "attention.cuh"
#include "gemm.cuh"
#include "small_kernels.cuh"

namespace dllm {

enum PhaseKind : int { PH_EMBED = 0, PH_GEMM = 1, PH_ATTN = 2, PH_MERGE = 3 };

struct StepPhase {
  int kind;
  int gemm_kind;
  int map_a, map_b, map_blo;   // indices into StepArgs::maps
  int layer;                   // attention: cache layer
  GemmParams g;
};

struct StepArgs {
  const StepPhase* phases;
  int n_phases;
  const CUtensorMap* maps;     // global memory, 64-byte aligned, written before the launch
  unsigned int* bar;           // grid arrival counter, zero at launch
  int* err;
  EmbedParams emb;
  AttnParams attn;             // z_k0 / z_v0 set per phase from its layer
  int attn_map;                // the K/V cache map
  int attn_items;              // b * H * q_tiles * splits
  MergeParams merge;
  unsigned long long* timeline;  // optional [grid][n_phases][6] (diagnostics), or null
  int prefetch;                  // weight tiles loaded ahead of a phase's barrier (<= ring depth)
};

template <int BN, int HD>
struct StepCfg {
  static constexpr int B_ROWS = BN <= 128 ? 2 * BN : BN;
  static constexpr int A_BYTES = 128 * 64 * 2;           // one weight tile (128 rows x 64 k)
  static constexpr int B_BYTES = B_ROWS * 64 * 2;        // one activation tile (hi and lo rows)
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ATT_KT = 32;                      // keys per attention tile
  static constexpr int ATT_TILE = ATT_KT * HD * 2;        // one of K, K lo, V, V lo
  static constexpr int XCH_BYTES = 128 * 33 * 4;         // epilogue exchange; also attention xo, merge arrays
  static constexpr int FIXED = 1024 + XCH_BYTES + 512 + 512 + 512;   // + row factors, params, barriers
  static constexpr int MAX_SMEM = 232448;
  static constexpr int ST_FIT = (MAX_SMEM - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = ST_FIT > 12 ? 12 : ST_FIT;
  // attention K/V tiles (with their low halves) borrow the activation half of
  // the ring, idle in ATTN phases
  static constexpr int AST = (STAGES * B_BYTES) / (4 * ATT_TILE) >= 2 ? 2 : 1;
  static constexpr int TMEM_COLS = 2 * B_ROWS;
  static constexpr int SMEM_BYTES = FIXED + STAGES * STAGE_BYTES;
  static_assert(STAGES >= 4, "ring too shallow");
  static_assert(AST * 4 * ATT_TILE <= STAGES * B_BYTES, "attention tiles fit the activation half of the ring");
  static_assert(32 * HD * 4 + 64 * 4 <= XCH_BYTES, "attention scratch");
  static_assert(sizeof(GemmParams) <= 512, "phase parameter copy");
  static_assert(BN <= 128, "persistent step: at most 128 activation rows per tile");
};

// ---------------------------------------------------------------- grid barrier
// Called by one thread after a CTA barrier over the workers.
__device__ __forceinline__ void grid_arrive(unsigned int* bar) {
  asm volatile("fence.proxy.async.global;" ::: "memory");   // our generic writes before others' TMA reads
  red_add_release_gpu(bar, 1u);
}

// Wait until `target` arrivals are counted; bounded by kWaitLimitNs.
__device__ __forceinline__ bool grid_wait(const unsigned int* bar, unsigned int target, volatile int* abort,
                                          int* err) {
  const unsigned long long t0 = globaltimer();
  for (;;) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
    if (v >= target) break;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_error(err, ERR_GRID_BARRIER);
      return false;
    }
    __nanosleep(256);   // ~300 pollers on one word: keep its L2 slice free for real traffic
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");   // later TMA reads see what the barrier published
  return true;
}

// ---------------------------------------------------------------- worker phases
// Embedding of rows r = first, first + stride, ... by 128 threads: the same
// per-element arithmetic and per-128-column reduction as embed_kernel.
__device__ __forceinline__ void embed_rows(const EmbedParams& p, int n_rows, int first, int stride, int tid) {
  for (int r = first; r < n_rows; r += stride) {
    const int seq = r / p.R, pos = p.row0 + r % p.R;
    const int tok = p.x[(long long)seq * p.T + pos];
    for (int c0 = tid * 8; c0 < p.d; c0 += 128 * 8) {
      const uint4 e = *reinterpret_cast<const uint4*>(p.embed + (long long)tok * p.d + c0);
      const uint4 gg = *reinterpret_cast<const uint4*>(p.g + c0);
      const uint16_t* ev = reinterpret_cast<const uint16_t*>(&e);
      const uint16_t* gv = reinterpret_cast<const uint16_t*>(&gg);
      float hv[8];
      uint16_t ov[8], lv[8];
      float sq = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        hv[i] = bf16_bits_to_f32(ev[i]);
        const float xv = hv[i] * bf16_bits_to_f32(gv[i]);
        ov[i] = f32_to_bf16_bits(xv);
        lv[i] = f32_to_bf16_bits(xv - bf16_bits_to_f32(ov[i]));
        sq += hv[i] * hv[i];
      }
      float4* hp = reinterpret_cast<float4*>(p.h + (long long)r * p.d + c0);
      hp[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
      hp[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
      *reinterpret_cast<uint4*>(p.xn + (long long)r * p.d + c0) = *reinterpret_cast<const uint4*>(ov);
      if (p.xn_lo)
        *reinterpret_cast<uint4*>(p.xn_lo + (long long)r * p.d + c0) = *reinterpret_cast<const uint4*>(lv);
#pragma unroll
      for (int s = 8; s >= 1; s >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, s);
      if ((tid & 15) == 0) p.ss[(long long)r * (p.d >> 7) + (c0 >> 7)] = sq;
    }
  }
}

// Merge of the LM-head tile statistics of one block row by 128 threads; the
// last row of a sequence to finish selects and commits for the sequence.
__device__ __forceinline__ void merge_row(const MergeParams& p, int row, int tid, uint8_t* scratch, int* flag) {
  MaxSumArg* part = reinterpret_cast<MaxSumArg*>(scratch);            // [4]
  float* conf_s = reinterpret_cast<float*>(scratch + 64);             // [256]
  int* arg_s = reinterpret_cast<int*>(scratch + 64 + 1024);
  int* rank_s = reinterpret_cast<int*>(scratch + 64 + 2048);
  float* eps_s = reinterpret_cast<float*>(scratch + 64 + 3072);
  int* best = reinterpret_cast<int*>(scratch + 64 + 4096);
  const int seq = row / p.B;
  const int warp = tid >> 5, lane = tid & 31;
  MaxSumArg acc{-INFINITY, 0.0f, 0x7fffffff};
  for (int t = tid; t < p.v_tiles; t += 128) {
    const long long o = (long long)t * p.n_rows + row;
    acc = msa_merge(acc, MaxSumArg{__ldcg(&p.st_m[o]), __ldcg(&p.st_s[o]), __ldcg(&p.st_a[o])});
  }
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    MaxSumArg o{__shfl_xor_sync(0xffffffffu, acc.m, s), __shfl_xor_sync(0xffffffffu, acc.s, s),
                __shfl_xor_sync(0xffffffffu, acc.a, s)};
    acc = (lane & s) ? msa_merge(o, acc) : msa_merge(acc, o);
  }
  if (lane == 0) part[warp] = acc;
  named_bar_sync(1, 128);
  if (tid == 0) {
    MaxSumArg r = part[0];
    for (int w = 1; w < 4; ++w) r = msa_merge(r, part[w]);
    p.conf[row] = 1.0f / r.s;
    p.arg[row] = r.a;
    const int old = atomic_add_acq_rel_gpu(&p.seq_done[seq], 1);
    *flag = (old == p.B - 1);
    if (*flag) p.seq_done[seq] = 0;
  }
  named_bar_sync(1, 128);
  if (!*flag) return;
  for (int i = tid; i < p.B; i += 128) {
    conf_s[i] = __ldcg(&p.conf[(long long)seq * p.B + i]);
    arg_s[i] = __ldcg(&p.arg[(long long)seq * p.B + i]);
  }
  named_bar_sync(1, 128);
  select_commit_group(conf_s, arg_s, rank_s, eps_s, p.B, p.x + (long long)seq * p.T + p.blk_start, p.mask_id,
                      p.rule, p.count + seq, best, tid, 128, [] { named_bar_sync(1, 128); });
  named_bar_sync(1, 128);
}

// ---------------------------------------------------------------- the kernel
template <int BN, int HD>
__global__ void __launch_bounds__(192, 1) step_kernel(const StepArgs a) {
  using C = StepCfg<BN, HD>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                        // STAGES weight tiles
  uint8_t* sB = sA + STAGES * C::A_BYTES;                    // STAGES activation tiles; attention K/V in ATTN phases
  float* xch = reinterpret_cast<float*>(sB + STAGES * C::B_BYTES);
  float* red = xch;                                          // RESID / LMHEAD never use xch at the same time
  float* rs_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xch) + C::XCH_BYTES);
  GemmParams* ps = reinterpret_cast<GemmParams*>(rs_s + 128);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(ps) + 512);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* afull = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(afull + C::AST);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bcast = reinterpret_cast<int*>(tmem_slot + 2);
  int* abcast = reinterpret_cast<int*>(tmem_slot + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x, cta = blockIdx.x;
  unsigned long long* tl = a.timeline ? a.timeline + cta * a.n_phases * 6 : nullptr;
  if (tl && threadIdx.x == 0) tl[1] = globaltimer();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    for (int s = 0; s < C::AST; ++s) mbar_init(&afull[s], 1);
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

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      // Walks this CTA's chunks of every GEMM phase in order through one ring.
      // At a phase's start it first loads the weight tiles of up to STAGES
      // chunks (they depend on nothing: the ring slots free up as the MMA
      // finishes the previous phase), then waits until every CTA finished the
      // previous phase and loads the matching activation tiles.
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      long long ring = 0;   // chunks issued so far, over all phases
      for (int ph = 0; ph < a.n_phases && !*abort_flag; ++ph) {
        const StepPhase& P = a.phases[ph];
        if (P.kind != PH_GEMM) continue;
        const long long total = P.g.total;
        const int kc = P.g.kc, n_tiles = P.g.n_tiles;
        const bool split = BN <= 128 && P.g.split != 0;
        const uint32_t tx = (uint32_t)(C::A_BYTES + (split ? 2 : 1) * BN * 128);
        const CUtensorMap* tA = a.maps + P.map_a;
        const CUtensorMap* tB = a.maps + P.map_b;
        const CUtensorMap* tBl = a.maps + P.map_blo;
        const long long start = cta * total / G, end = (cta + 1) * total / G;
        const long long n = end - start;
        const long long depth = a.prefetch < STAGES ? a.prefetch : STAGES;
        const long long pre = n < depth ? n : depth;
        bool ok = true;
        for (long long i = 0; i < pre && ok; ++i) {
          const long long c = ring + i;
          const int s = (int)(c % STAGES);
          if (!mbar_wait(&empty[s], (uint32_t)(((c / STAGES) & 1) ^ 1), abort_flag, a.err, ERR_GEMM_EMPTY)) {
            ok = false;
            break;
          }
          const long long gch = start + i;
          const long long tile = gch / kc;
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(sA + s * C::A_BYTES, tA, &full[s], (int)(gch - tile * kc) * 64, (int)(tile / n_tiles) * 128,
                      pol_w);
        }
        if (!ok) break;
        if (!grid_wait(a.bar, (unsigned int)(G * ph), abort_flag, a.err)) break;
        if (tl) tl[ph * 6 + 1] = globaltimer();
        for (long long i = 0; i < pre; ++i) {
          const long long c = ring + i;
          const int s = (int)(c % STAGES);
          const long long gch = start + i;
          const long long tile = gch / kc;
          const int k = (int)(gch - tile * kc), n_idx = (int)(tile % n_tiles);
          tma_load_2d(sB + s * C::B_BYTES, tB, &full[s], k * 64, n_idx * BN, pol_x);
          if (split) tma_load_2d(sB + s * C::B_BYTES + BN * 128, tBl, &full[s], k * 64, n_idx * BN, pol_x);
        }
        for (long long i = pre; i < n; ++i) {
          const long long c = ring + i;
          const int s = (int)(c % STAGES);
          if (!mbar_wait(&empty[s], (uint32_t)(((c / STAGES) & 1) ^ 1), abort_flag, a.err, ERR_GEMM_EMPTY)) {
            ok = false;
            break;
          }
          const long long gch = start + i;
          const long long tile = gch / kc;
          const int k = (int)(gch - tile * kc), n_idx = (int)(tile % n_tiles), m_idx = (int)(tile / n_tiles);
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(sA + s * C::A_BYTES, tA, &full[s], k * 64, m_idx * 128, pol_w);
          tma_load_2d(sB + s * C::B_BYTES, tB, &full[s], k * 64, n_idx * BN, pol_x);
          if (split) tma_load_2d(sB + s * C::B_BYTES + BN * 128, tBl, &full[s], k * 64, n_idx * BN, pol_x);
        }
        if (!ok) break;
        if (tl) tl[ph * 6 + 3] = globaltimer();
        ring += n;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      long long ring = 0;
      int seg = 0;
      bool ok = true;
      for (int ph = 0; ph < a.n_phases && ok; ++ph) {
        const StepPhase& P = a.phases[ph];
        if (P.kind != PH_GEMM) continue;
        const long long total = P.g.total;
        const int kc = P.g.kc;
        const bool split = BN <= 128 && P.g.split != 0;
        const uint32_t idesc = idesc_bf16_f32(128, split ? 2 * BN : BN);
        const long long start = cta * total / G, end = (cta + 1) * total / G;
        long long g = start;
        while (g < end) {
          const long long tile = g / kc;
          const long long seg_first = g;
          const long long seg_end = ((tile + 1) * kc < end) ? (tile + 1) * kc : end;
          const int buf = seg & 1;
          const uint32_t use = (uint32_t)(seg >> 1);
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, a.err, ERR_GEMM_TEMPTY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * C::B_ROWS);
          for (; g < seg_end; ++g, ++ring) {
            const int s = (int)(ring % STAGES);
            if (!mbar_wait(&full[s], (uint32_t)((ring / STAGES) & 1), abort_flag, a.err, ERR_GEMM_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * C::A_BYTES);
            const uint32_t b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc,
                          (g > seg_first || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
          }
          if (!ok) break;
          mma_commit(&tfull[buf]);
          ++seg;
        }
        if (tl) tl[ph * 6 + 2] = globaltimer();
      }
    }
  } else {
    // -------------------------------------------------- workers (warps 2..5)
    const int q = warp & 3;
    const int l128 = q * 32 + lane;
    int seg = 0;
    uint32_t att_tc = 0;
    for (int ph = 0; ph < a.n_phases; ++ph) {
      if (ph > 0) {
        if (l128 == 0) grid_wait(a.bar, (unsigned int)(G * ph), abort_flag, a.err);
        if (named_bar_or(1, 128, *abort_flag != 0)) break;
      }
      if (tl && l128 == 0) tl[ph * 6 + 4] = globaltimer();
      const StepPhase& P = a.phases[ph];
      if (P.kind == PH_EMBED) {
        embed_rows(a.emb, a.merge.n_rows, (int)cta, (int)G, l128);
      } else if (P.kind == PH_ATTN) {
        AttnParams ap = a.attn;
        ap.z_k0 = ((P.layer * 2 + 0) * 2 + 0) * ap.b * ap.H;
        ap.z_kl0 = ((P.layer * 2 + 0) * 2 + 1) * ap.b * ap.H;
        ap.z_v0 = ((P.layer * 2 + 1) * 2 + 0) * ap.b * ap.H;
        ap.z_vl0 = ((P.layer * 2 + 1) * 2 + 1) * ap.b * ap.H;
        const CUtensorMap* tkv = a.maps + a.attn_map;
        uint8_t* sK = sB;                                    // the activation half of the ring is idle now
        uint8_t* sV = sB + C::AST * 2 * C::ATT_TILE;
        for (int item = (int)cta; item < a.attn_items; item += (int)G) {
          const int split = item % ap.splits;
          const int rest = item / ap.splits;
          const int qt = rest % ap.q_tiles;
          const int head = (rest / ap.q_tiles) % ap.H;
          const int sq = rest / (ap.q_tiles * ap.H);
          attn_item<HD, 2, C::AST, C::ATT_KT>(tkv, tkv, ap, split, qt, head, sq, sK, sV, xch, afull, abcast, att_tc,
                                              l128);
          named_bar_sync(2, 128);
        }
      } else if (P.kind == PH_MERGE) {
        for (int row = (int)cta; row < a.merge.n_rows; row += (int)G)
          merge_row(a.merge, row, l128, reinterpret_cast<uint8_t*>(xch), bcast);
      } else {
        // GEMM epilogue over this CTA's segments of the phase; the phase's
        // parameters are copied to shared memory
        for (int w = l128; w < (int)(sizeof(GemmParams) / 4); w += 128)
          reinterpret_cast<int*>(ps)[w] = reinterpret_cast<const int*>(&P.g)[w];
        named_bar_sync(1, 128);
        const GemmParams& p = *ps;
        const long long total = p.total;
        const int kc = p.kc, n_tiles = p.n_tiles;
        const bool split = BN <= 128 && p.split != 0;
        const long long start = cta * total / G, end = (cta + 1) * total / G;
        long long g = start;
        bool stop = false;
        int rs_tile = -1;
        while (g < end && !stop) {
          const long long tile = g / kc;
          const long long seg_first = g;
          const long long seg_end = ((tile + 1) * kc < end) ? (tile + 1) * kc : end;
          const bool full_tile = (seg_first == tile * kc) && (seg_end == (tile + 1) * kc);
          const int m_idx = (int)(tile / n_tiles);
          const int n_idx = (int)(tile % n_tiles);
          const int buf = seg & 1;
          const uint32_t use = (uint32_t)(seg >> 1);
          if (n_idx != rs_tile) {
            // RMSNorm row factors of this activation tile: stage the partial
            // sums of squares in smem with parallel loads, then each column
            // sums its partials in order
            rs_tile = n_idx;
            named_bar_sync(1, 128);
            if (p.ss_in) {
              const int tiles = p.ss_in_tiles;
              for (int c0 = 0; c0 < BN; c0 += 32) {
                for (int e = l128; e < 32 * tiles; e += 128) {
                  const int c = e / tiles, t = e - c * tiles;
                  const int r = n_idx * BN + c0 + c;
                  xch[e] = r < p.N ? __ldcg(&p.ss_in[(long long)r * tiles + t]) : 0.0f;
                }
                named_bar_sync(1, 128);
                if (l128 < 32) {
                  const int r = n_idx * BN + c0 + l128;
                  float sum = 0.0f;
                  for (int t = 0; t < tiles; ++t) sum += xch[l128 * tiles + t];
                  rs_s[c0 + l128] = r < p.N ? rsqrtf(sum * p.inv_d + p.eps) : 0.0f;
                }
                named_bar_sync(1, 128);
              }
            } else {
              for (int c = l128; c < BN; c += 128) rs_s[c] = 1.0f;
            }
            named_bar_sync(1, 128);
          }
          mbar_wait(&tfull[buf], use & 1u, abort_flag, a.err, ERR_GEMM_TFULL);
          if (named_bar_or(1, 128, *abort_flag != 0)) {
            stop = true;
            break;
          }
          if (tl && l128 == 0 && g == start) tl[ph * 6 + 5] = globaltimer();
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
              switch (P.gemm_kind) {
                case GEMM_QKV: epi_chunk<GEMM_QKV>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                case GEMM_RESID: epi_chunk<GEMM_RESID>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                case GEMM_SWIGLU: epi_chunk<GEMM_SWIGLU>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                default: epi_chunk<GEMM_LMHEAD>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
              }
            }
          } else {
            const int slot = (seg_first == start) ? 0 : 1;
            float* wsp = p.ws + ((cta * 2 + slot) * (long long)BN) * 128;
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
            const long long t0 = tile * kc, t1 = (tile + 1) * kc - 1;
            const long long c_first = sk_owner(t0, G, total), c_last = sk_owner(t1, G, total);
            if (l128 == 0) {
              // contributors: the CTAs in [c_first, c_last] whose chunk range is not
          // empty (with fewer chunks than CTAs some ranges are)
          int contributors = 0;
          for (long long ctr = c_first; ctr <= c_last; ++ctr)
            contributors += (ctr * total / G) < ((ctr + 1) * total / G) ? 1 : 0;
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
                for (long long ctr = c_first; ctr <= c_last; ++ctr) {
                  const long long st = ctr * total / G;
                  if (st == (ctr + 1) * total / G) continue;   // empty range: no partial
                  const long long sstart = st > t0 ? st : t0;
                  const int sl = (sstart == st) ? 0 : 1;
                  const float* src = p.ws + ((ctr * 2 + sl) * (long long)BN) * 128;
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] += __ldcg(&src[(long long)(c0 + j) * 128 + l128]);
                }
                switch (P.gemm_kind) {
                  case GEMM_QKV: epi_chunk<GEMM_QKV>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                  case GEMM_RESID: epi_chunk<GEMM_RESID>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                  case GEMM_SWIGLU: epi_chunk<GEMM_SWIGLU>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                  default: epi_chunk<GEMM_LMHEAD>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                }
              }
            }
          }
          g = seg_end;
          ++seg;
        }
        if (stop) break;
      }
      // publish this CTA's part of the phase
      named_bar_sync(1, 128);
      if (l128 == 0) {
        if (tl) tl[ph * 6] = globaltimer();
        grid_arrive(a.bar);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace dllm
