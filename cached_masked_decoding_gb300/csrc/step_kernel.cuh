// Persistent DualCache denoise step: one cooperative launch, one CTA per SM,
// runs every phase of a step - embedding, per layer [QKV+RoPE+K/V write,
// block attention, O-proj+residual+norm, gate/up+SwiGLU, down+residual+norm],
// LM head + softmax statistics, statistic merge + select/commit - ordered by
// dataflow flags instead of grid barriers: every finished unit of a phase (a
// GEMM row tile, an attention head) raises a counter, and a consumer waits
// only for the units it reads (waits bounded in time).
//
// Why: a DualCache step streams ~15 GB of weights through 160 GEMM phases of
// 5-30 us each.  As separate launches every phase pays a pipeline fill (the
// first TMA tile lands ~3 us after the CTA starts) and an epilogue tail.  Here
// the TMA producer walks straight from one GEMM phase into the next: it keeps
// loading the next phase's weight tiles into the shared-memory ring (weights
// depend on nothing) while the other CTAs finish the current phase's
// epilogues, and each activation tile waits only for the row tile or head
// that writes its 64 columns - so a phase starts on the columns that are
// ready while the previous phase's last tiles are still being reduced.
//
// Ordering.  A unit's finisher writes its outputs, passes a barrier of the
// four epilogue warps, and one thread raises the unit's flag with a release
// (after a proxy fence, as the readers are TMA loads); readers acquire it.
// Buffers reused across phases stay safe without barriers because every
// GEMM reads all of its input columns: a unit of phase p+2 can only start
// after all of phase p+1's units finished, hence after all of phase p's
// readers.  The stream-K partial workspace alternates between two halves by
// GEMM phase for the same reason.
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

// Diagnostic timeline slots per (CTA, phase), %globaltimer ns:
// 0 workers finished the phase, 1 producer issued the phase's first
// activation tile (phase 0: kernel start), 2 MMA issuer finished the phase,
// 3 producer issued the phase's last tile, 4 workers started the phase,
// 5 workers got the phase's first accumulator, 6 workers were through their
// first segment, 7 workers started their last fix-up as the last
// contributor, 8 it had summed the partials, 9 workers published their last
// unit of the phase.  Attention phases: 5 first item's inputs ready, 6 first
// item done, 7 its keys done, 8 its split partial stored and counted, 9 last
// head published by this CTA.
constexpr int kTimelineSlots = 10;

struct StepPhase {
  int kind;
  int gemm_kind;
  int map_a, map_b, map_blo;   // indices into StepArgs::maps
  int layer;                   // attention: cache layer
  // dataflow (indices into StepArgs::flags)
  int unit0;     // first flag of this phase's units: GEMM row tiles (count n-tiles) or attention heads (count works)
  int done;      // counter of this phase's finished units (GEMM tiles, attention works, CTAs for the embedding)
  int dep0;      // first flag of the units that write this phase's activation columns
  int dep_shift; // activation k-chunk (64 columns) k is written by unit k >> dep_shift
  int dep_need;  // value such a unit's flag reaches when it is complete
  int dep_attn;  // 1: the activations are the attention output of this layer (attention uses the ring's B half)
  int rs_done;   // counter that must reach rs_need before the row factors / the merge may read (-1: none)
  int rs_need;
  int src_done, src_need;   // completion counter of the phase producing the activations, and its final value
  int qkv0;      // attention: first row-tile flag of this layer's QKV phase
  int qkv_need;  // value a QKV row-tile flag reaches when complete
  GemmParams g;
};

struct StepArgs {
  const StepPhase* phases;
  int n_phases;
  const CUtensorMap* maps;     // global memory, 64-byte aligned, written before the launch
  int* flags;                  // dataflow flags and counters, zero at launch
  int* err;
  EmbedParams emb;
  AttnParams attn;             // z_k0 / z_v0 set per phase from its layer
  int attn_map;                // the K/V cache map
  int attn_items;              // b * H * q_tiles * splits
  MergeParams merge;
  unsigned long long* timeline;  // optional [grid][n_phases][kTimelineSlots] (diagnostics), or null
  int prefetch;                  // weight tiles loaded ahead of a phase's barrier (<= ring depth)
  int skip_done;                 // 1: do nothing when the block [merge.blk_start, + merge.B) of every sequence holds no MASK
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
  // with 32 activation rows, the residual rows of a RESID tile (32 x 128
  // floats) fit in the shared memory left over: they are copied there while
  // the tile's MMAs stream, so the epilogue does not wait for L2 reads
  static constexpr int H_BYTES = 32 * 128 * 4;
  static constexpr bool H_PRE = BN == 32 && FIXED + STAGES * STAGE_BYTES + H_BYTES <= MAX_SMEM;
  static constexpr int SMEM_BYTES = FIXED + STAGES * STAGE_BYTES + (H_PRE ? H_BYTES : 0);
  static_assert(STAGES >= 4, "ring too shallow");
  static_assert(AST * 4 * ATT_TILE <= STAGES * B_BYTES, "attention tiles fit the activation half of the ring");
  static_assert(32 * HD * 4 + 64 * 4 <= XCH_BYTES, "attention scratch");
  static_assert(sizeof(GemmParams) <= 512, "phase parameter copy");
  static_assert(BN <= 128, "persistent step: at most 128 activation rows per tile");
};

// ---------------------------------------------------------------- dataflow flags
__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until *f >= need (acquire), then order later TMA reads after it.
// Bounded by limit_ns; gives up early once this CTA raised *abort or any
// CTA recorded an error; on giving up records `site` in err.  The poll is
// one acquire load per round trip (one thread per CTA polls); the error word
// and the clock are looked at every 16th round, so a flag raised between
// two polls is seen one L2 round trip later at most.
__device__ __forceinline__ bool flag_wait_for(const int* f, int need, volatile int* abort, int* err,
                                              unsigned long long limit_ns, int site) {
  if (ld_acquire_gpu(f) < need) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
      if (ld_acquire_gpu(f) >= need) break;
      if ((i & 15u) == 0) {
        if (*abort || ld_relaxed_gpu(err) != 0) {
          *abort = 1;
          return false;
        }
        if (globaltimer() - t0 > limit_ns) {
          *abort = 1;
          record_error(err, site);
          return false;
        }
      }
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__device__ __forceinline__ bool flag_wait(const int* f, int need, volatile int* abort, int* err) {
  return flag_wait_for(f, need, abort, err, kWaitLimitNs, ERR_STEP_FLAG);
}

// Wait until *f0 >= need0 and *f1 >= need1 (f1 may be null).  The first
// look reads both with relaxed loads issued together (one round trip) and
// turns them into an acquire with a fence; only a flag not yet raised is
// then polled.
__device__ __forceinline__ bool flags_wait2(const int* f0, int need0, const int* f1, int need1,
                                            volatile int* abort, int* err) {
  const int v0 = ld_relaxed_gpu(f0);
  const int v1 = f1 ? ld_relaxed_gpu(f1) : need1;
  if (v0 >= need0 && v1 >= need1) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
  }
  if (v0 < need0 && !flag_wait(f0, need0, abort, err)) return false;
  if (f1 && v1 < need1 && !flag_wait(f1, need1, abort, err)) return false;
  asm volatile("fence.acq_rel.gpu;" ::: "memory");   // also covers the flag seen by the relaxed load
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// Raise two counters by one with release semantics.  Called by one thread
// after a barrier over the threads whose writes it publishes; the proxy fence
// makes those writes visible to other CTAs' TMA reads.  One acq_rel fence
// followed by two relaxed reductions releases both (two release reductions
// would wait for the stores twice: about 0.6 us each).
__device__ __forceinline__ void flag_publish(int* a, int* b) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(a) : "memory");
  if (b) asm volatile("red.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(b) : "memory");
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
  if (a.skip_done) {
    // launched before the host saw the previous step's commits: if that step
    // finished the block there is nothing to denoise, and the launch ends
    // here, before any write (every CTA reaches the same answer)
    const int n = a.attn.b * a.merge.B;
    int masked = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int sq = i / a.merge.B, c = i - sq * a.merge.B;
      masked |= a.merge.x[(long long)sq * a.merge.T + a.merge.blk_start + c] == a.merge.mask_id;
    }
    if (!__syncthreads_or(masked)) return;
  }
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
  volatile int* att_done = reinterpret_cast<volatile int*>(tmem_slot + 4);   // layers whose attention items this CTA finished
  float* hs = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xch) + C::XCH_BYTES + 1536);   // [32][128] (H_PRE)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x, cta = blockIdx.x;
  unsigned long long* tl = a.timeline ? a.timeline + cta * a.n_phases * kTimelineSlots : nullptr;
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
    *att_done = 0;
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
      // finishes the previous phase), then loads each chunk's activation tile
      // once the unit writing those 64 columns has finished.
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      RingPos rw{0, 0u};   // ring position of the next weight load, over all phases
      for (int ph = 0; ph < a.n_phases && !*abort_flag; ++ph) {
        const StepPhase& P = a.phases[ph];
        if (P.kind != PH_GEMM) continue;
        const uint32_t total = (uint32_t)P.g.total;
        const int kc = P.g.kc, n_tiles = P.g.n_tiles;
        const bool split = BN <= 128 && P.g.split != 0;
        const uint32_t tx = (uint32_t)(C::A_BYTES + (split ? 2 : 1) * BN * 128);
        const CUtensorMap* tA = a.maps + P.map_a;
        const CUtensorMap* tB = a.maps + P.map_b;
        const CUtensorMap* tBl = a.maps + P.map_blo;
        const int* dep = a.flags + P.dep0;
        const int dep_shift = P.dep_shift, dep_need = P.dep_need;
        const uint32_t start = sk_begin((uint32_t)cta, (uint32_t)G, total);
        const int n = (int)(sk_begin((uint32_t)cta + 1, (uint32_t)G, total) - start);
        const int depth = a.prefetch < STAGES ? a.prefetch : STAGES;
        const int pre = n < depth ? n : depth;
        ChunkPos cw;
        cw.init(start, kc, n_tiles);
        const ChunkPos c_first = cw;
        const RingPos r_first = rw;
        bool ok = true;
        for (int i = 0; i < pre; ++i) {
          if (!mbar_wait(&empty[rw.s], rw.par ^ 1u, abort_flag, a.err, ERR_GEMM_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[rw.s], tx);
          tma_load_2d(sA + rw.s * C::A_BYTES, tA, &full[rw.s], cw.k * 64, cw.m * 128, pol_w);
          cw.next(kc, n_tiles);
          rw.next(STAGES);
        }
        if (!ok) break;
        if (P.dep_attn) {
          // the activation half of the ring holds this CTA's attention tiles
          // until its workers are through this layer's attention items
          const unsigned long long t0 = globaltimer();
          while (*att_done < P.layer + 1) {
            if (*abort_flag || globaltimer() - t0 > kWaitLimitNs) {
              if (!*abort_flag) record_error(a.err, ERR_STEP_LOCAL);
              *abort_flag = 1;
              ok = false;
              break;
            }
            __nanosleep(64);
          }
          if (!ok) break;
        }
        // activation columns [64k, 64k+64) come from unit k >> dep_shift.
        // Units [ready_lo, ready_hi] are known complete; a look reads the
        // flags of the unit a chunk needs and of the next three together (one
        // round trip: the chunks of a segment visit the units in ascending
        // order), and once the whole producing phase is seen complete nothing
        // is polled
        int ready_lo = 0, ready_hi = -1;
        bool all_ready = false;
        const int* src_done = a.flags + P.src_done;
        const int src_need = P.src_need;
        const int last_unit = dep_shift >= 31 ? 0 : (kc - 1) >> dep_shift;
        auto dep_ready = [&](int k) -> bool {
          if (all_ready) return true;
          const int unit = k >> dep_shift;
          if (unit >= ready_lo && unit <= ready_hi) return true;
          const int vd = ld_relaxed_gpu(src_done);
          int vu[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) vu[j] = unit + j <= last_unit ? ld_relaxed_gpu(dep + unit + j) : 0;
          int hi = unit;
          if (vd >= src_need) {
            all_ready = true;
          } else if (vu[0] < dep_need) {
            if (!flag_wait(dep + unit, dep_need, abort_flag, a.err)) return false;
            ready_lo = ready_hi = unit;
            return true;
          } else {
#pragma unroll
            for (int j = 1; j < 4; ++j)
              if (hi == unit + j - 1 && unit + j <= last_unit && vu[j] >= dep_need) hi = unit + j;
          }
          ready_lo = unit;
          ready_hi = hi;
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
          return true;
        };
        ChunkPos cx = c_first;
        RingPos rx = r_first;
        for (int i = 0; i < pre; ++i) {
          if (!dep_ready(cx.k)) {
            ok = false;
            break;
          }
          if (tl && i == 0) tl[ph * kTimelineSlots + 1] = globaltimer();
          tma_load_2d(sB + rx.s * C::B_BYTES, tB, &full[rx.s], cx.k * 64, cx.n * BN, pol_x);
          if (split) tma_load_2d(sB + rx.s * C::B_BYTES + BN * 128, tBl, &full[rx.s], cx.k * 64, cx.n * BN, pol_x);
          cx.next(kc, n_tiles);
          rx.next(STAGES);
        }
        for (int i = pre; i < n && ok; ++i) {
          if (!mbar_wait(&empty[rw.s], rw.par ^ 1u, abort_flag, a.err, ERR_GEMM_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[rw.s], tx);
          tma_load_2d(sA + rw.s * C::A_BYTES, tA, &full[rw.s], cw.k * 64, cw.m * 128, pol_w);
          if (!dep_ready(cw.k)) {
            ok = false;
            break;
          }
          tma_load_2d(sB + rw.s * C::B_BYTES, tB, &full[rw.s], cw.k * 64, cw.n * BN, pol_x);
          if (split) tma_load_2d(sB + rw.s * C::B_BYTES + BN * 128, tBl, &full[rw.s], cw.k * 64, cw.n * BN, pol_x);
          cw.next(kc, n_tiles);
          rw.next(STAGES);
        }
        if (!ok) break;
        if (tl) tl[ph * kTimelineSlots + 3] = globaltimer();
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      RingPos rm{0, 0u};
      int seg = 0;
      bool ok = true;
      for (int ph = 0; ph < a.n_phases && ok; ++ph) {
        const StepPhase& P = a.phases[ph];
        if (P.kind != PH_GEMM) continue;
        const uint32_t total = (uint32_t)P.g.total;
        const uint32_t kc = (uint32_t)P.g.kc;
        const bool split = BN <= 128 && P.g.split != 0;
        const uint32_t idesc = idesc_bf16_f32(128, split ? 2 * BN : BN);
        uint32_t g = sk_begin((uint32_t)cta, (uint32_t)G, total);
        const uint32_t end = sk_begin((uint32_t)cta + 1, (uint32_t)G, total);
        uint32_t k = g % kc;
        while (g < end) {
          const uint32_t len = (kc - k < end - g) ? kc - k : end - g;   // this segment: the rest of a tile
          const int buf = seg & 1;
          const uint32_t use = (uint32_t)(seg >> 1);
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, a.err, ERR_GEMM_TEMPTY)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(buf * C::B_ROWS);
          for (uint32_t i = 0; i < len; ++i) {
            if (!mbar_wait(&full[rm.s], rm.par, abort_flag, a.err, ERR_GEMM_FULL)) {
              ok = false;
              break;
            }
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
          g += len;
          k = 0;
        }
        if (tl) tl[ph * kTimelineSlots + 2] = globaltimer();
      }
    }
  } else {
    // -------------------------------------------------- workers (warps 2..5)
    const int q = warp & 3;
    const int l128 = q * 32 + lane;
    int seg = 0;
    uint32_t att_tc = 0;
    for (int ph = 0; ph < a.n_phases; ++ph) {
      const StepPhase& P = a.phases[ph];
      if (tl && l128 == 0) tl[ph * kTimelineSlots + 4] = globaltimer();
      // a phase that reads row statistics (or, for the merge, every LM-head
      // tile) waits until all units of the phase producing them finished
      if (P.rs_done >= 0 && l128 == 0) flag_wait(a.flags + P.rs_done, P.rs_need, abort_flag, a.err);
      if (named_bar_or(1, 128, *abort_flag != 0)) break;
      if (P.kind == PH_EMBED) {
        embed_rows(a.emb, a.attn.b * a.emb.R, (int)cta, (int)G, l128);
        named_bar_sync(1, 128);
        if (l128 == 0) flag_publish(a.flags + P.done, nullptr);
      } else if (P.kind == PH_ATTN) {
        AttnParams ap = a.attn;
        ap.z_k0 = ((P.layer * 2 + 0) * 2 + 0) * ap.b * ap.H;
        ap.z_kl0 = ((P.layer * 2 + 0) * 2 + 1) * ap.b * ap.H;
        ap.z_v0 = ((P.layer * 2 + 1) * 2 + 0) * ap.b * ap.H;
        ap.z_vl0 = ((P.layer * 2 + 1) * 2 + 1) * ap.b * ap.H;
        const CUtensorMap* tkv = a.maps + a.attn_map;
        uint8_t* sK = sB;                                    // the activation half of the ring is idle now
        uint8_t* sV = sB + C::AST * 2 * C::ATT_TILE;
        bool stop = false;
        for (int item = (int)cta; item < a.attn_items; item += (int)G) {
          const int split = item % ap.splits;
          const int rest = item / ap.splits;
          const int qt = rest % ap.q_tiles;
          const int head = (rest / ap.q_tiles) % ap.H;
          const int sq = rest / (ap.q_tiles * ap.H);
          if (l128 == 0) {
            // q, k and v of this head: the QKV row tiles holding its columns
            const int d = ap.H * HD, c0 = head * HD;
            if (flags_wait2(a.flags + P.qkv0 + c0 / 128, P.qkv_need, a.flags + P.qkv0 + (d + c0) / 128, P.qkv_need,
                            abort_flag, a.err))
              flags_wait2(a.flags + P.qkv0 + (2 * d + c0) / 128, P.qkv_need, nullptr, 0, abort_flag, a.err);
          }
          if (named_bar_or(1, 128, *abort_flag != 0)) {
            stop = true;
            break;
          }
          const bool first = item == (int)cta;
          if (tl && l128 == 0 && first) tl[ph * kTimelineSlots + 5] = globaltimer();
          const bool fin = attn_item<HD, 2, C::AST, C::ATT_KT>(tkv, tkv, ap, split, qt, head, sq, sK, sV, xch, afull,
                                                               abcast, att_tc, l128,
                                                               tl && first ? tl + ph * kTimelineSlots + 7 : nullptr);
          named_bar_sync(2, 128);
          if (fin && l128 == 0) flag_publish(a.flags + P.unit0 + head, a.flags + P.done);
          if (tl && l128 == 0) {
            if (first) tl[ph * kTimelineSlots + 6] = globaltimer();
            if (fin) tl[ph * kTimelineSlots + 9] = globaltimer();
          }
        }
        if (stop) break;
        if (l128 == 0) *att_done = P.layer + 1;
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
        const uint32_t total = (uint32_t)p.total, uG = (uint32_t)G;
        const int kc = p.kc, n_tiles = p.n_tiles;
        const bool split = BN <= 128 && p.split != 0;
        const uint32_t start = sk_begin((uint32_t)cta, uG, total), end = sk_begin((uint32_t)cta + 1, uG, total);
        // RESID: the first tile whose epilogue this CTA runs (the first tile
        // starting in its range) has its residual rows copied to shared memory
        // now; they were written by an earlier phase whose completion this
        // CTA's workers have already acquired
        int h_tile = -1;
        if constexpr (C::H_PRE) {
          if (P.gemm_kind == GEMM_RESID) {
            const uint32_t tf = (start + (uint32_t)kc - 1) / (uint32_t)kc;
            if (tf * (uint32_t)kc < end) {
              h_tile = (int)tf;
              const int hm = h_tile / n_tiles, hr0 = (h_tile - hm * n_tiles) * BN;
              for (int e = l128; e < 32 * 32; e += 128) {
                const int row = e >> 5, c4 = (e & 31) * 4;
                if (hr0 + row < p.N)
                  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(hs + row * 128 + c4)),
                               "l"(p.h + (long long)(hr0 + row) * p.d_model + hm * 128 + c4)
                               : "memory");
              }
              asm volatile("cp.async.commit_group;" ::: "memory");
            }
          }
        }
        uint32_t g = start;
        ChunkPos cp;
        cp.init(start, kc, n_tiles);
        bool stop = false;
        int rs_tile = -1;
        while (g < end && !stop) {
          const uint32_t len = ((uint32_t)(kc - cp.k) < end - g) ? (uint32_t)(kc - cp.k) : end - g;
          const uint32_t seg_end = g + len;
          const uint32_t t0 = g - (uint32_t)cp.k;            // first chunk of this tile
          const bool full_tile = (cp.k == 0) && (len == (uint32_t)kc);
          const int m_idx = cp.m;
          const int n_idx = cp.n;
          const int tile = m_idx * n_tiles + n_idx;
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
          if (tl && l128 == 0 && g == start) tl[ph * kTimelineSlots + 5] = globaltimer();
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
                case GEMM_RESID: epi_chunk<GEMM_RESID>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red, tile == h_tile ? hs : nullptr); break;
                case GEMM_SWIGLU: epi_chunk<GEMM_SWIGLU>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                default: epi_chunk<GEMM_LMHEAD>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
              }
            }
            named_bar_sync(1, 128);
            if (l128 == 0) flag_publish(a.flags + P.unit0 + m_idx, a.flags + P.done);
            if (tl && l128 == 0) {
              if (g == start) tl[ph * kTimelineSlots + 6] = globaltimer();
              tl[ph * kTimelineSlots + 9] = globaltimer();
            }
          } else {
            // A tile cut between CTAs is owned by the CTA whose range holds
            // its first chunk.  The other contributors store their partial
            // and count in; the owner keeps its own sums in tensor memory,
            // waits until the others have counted in, adds their partials in
            // contributor order and runs the epilogue.  A CTA owns at most the
            // one tile that starts in its range, so no CTA runs two
            // reductions back to back, and the owner's own partial never
            // leaves the SM.
            const uint32_t t1 = t0 + (uint32_t)kc - 1;
            const uint32_t c_first = sk_owner32(t0, uG, total), c_last = sk_owner32(t1, uG, total);
            if (g != t0) {
              // a contributor's segment in a tile it does not own is the first
              // of its range: one partial slot per CTA
              // stored through shared memory as [rows][128 features], 16 bytes
              // per thread and store
              float* wsp = p.ws + ((cta * 2) * (long long)BN) * 128;
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
                named_bar_sync(1, 128);
#pragma unroll
                for (int c = 0; c < 32; ++c) xch[c * kStageLd + l128] = v[c];
                named_bar_sync(1, 128);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int row = q + 4 * k;
                  __stcg(reinterpret_cast<float4*>(&wsp[(long long)(c0 + row) * 128 + lane * 4]),
                         *reinterpret_cast<const float4*>(xch + row * kStageLd + lane * 4));
                }
              }
              named_bar_sync(1, 128);
              if (l128 == 0) {
                // the owner reads the partial with generic loads: a release suffices
                asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(&p.counters[tile]) : "memory");
                if (tl && g == start) tl[ph * kTimelineSlots + 6] = globaltimer();
              }
            } else {
              if (l128 == 0) {
                // the other contributors: CTAs in (c_first, c_last] whose chunk
                // range is not empty (with fewer chunks than CTAs some are)
                int others = 0;
                uint32_t st = sk_begin(c_first + 1, uG, total);
                for (uint32_t ctr = c_first + 1; ctr <= c_last; ++ctr) {
                  const uint32_t en = sk_begin(ctr + 1, uG, total);
                  others += st < en ? 1 : 0;
                  st = en;
                }
                if (tl) tl[ph * kTimelineSlots + 7] = globaltimer();
                flag_wait(&p.counters[tile], others, abort_flag, a.err);
              }
              if (named_bar_or(1, 128, *abort_flag != 0)) {
                stop = true;
                break;
              }
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
                // the others' partials in contributor order, two at a time so
                // that both sets of loads are in flight: ((own + p1) + p2) + ...
                uint32_t ctr = c_first + 1;
                uint32_t st = sk_begin(c_first + 1, uG, total);
                while (ctr <= c_last) {
                  const float* src0 = nullptr;
                  const float* src1 = nullptr;
                  int ns = 0;
                  for (; ctr <= c_last && ns < 2; ++ctr) {
                    const uint32_t en = sk_begin(ctr + 1, uG, total);
                    const uint32_t cst = st;
                    st = en;
                    if (cst == en) continue;                     // empty range: no partial
                    const float* sp = p.ws + (((long long)ctr * 2) * BN) * 128 + (long long)c0 * 128 + l128;
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
                if (tl && l128 == 0 && c0 == 0) tl[ph * kTimelineSlots + 8] = globaltimer();
                switch (P.gemm_kind) {
                  case GEMM_QKV: epi_chunk<GEMM_QKV>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                  case GEMM_RESID: epi_chunk<GEMM_RESID>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red, tile == h_tile ? hs : nullptr); break;
                  case GEMM_SWIGLU: epi_chunk<GEMM_SWIGLU>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                  default: epi_chunk<GEMM_LMHEAD>(p, v, m_idx, n_idx * BN + c0, l128, lane, q, xch, rs_s + c0, red); break;
                }
              }
              named_bar_sync(1, 128);
              if (l128 == 0) flag_publish(a.flags + P.unit0 + m_idx, a.flags + P.done);
              if (tl && l128 == 0) tl[ph * kTimelineSlots + 9] = globaltimer();
            }
          }
          g = seg_end;
          cp.k = 0;                                            // the next segment starts a tile
          if (++cp.n == n_tiles) {
            cp.n = 0;
            ++cp.m;
          }
          ++seg;
        }
        if (h_tile >= 0) asm volatile("cp.async.wait_all;" ::: "memory");
        if (stop) break;
      }
      if (tl && l128 == 0) tl[ph * kTimelineSlots] = globaltimer();
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
