// Embedding gather, LM-head statistic merge and the select/commit rule.
#pragma once

#include "ptx.cuh"

namespace dllm {

// ------------------------------------------------------------------ embedding
// h[r] = E[x[seq][row0 + r % R]] (f32), xn[r] = bf16(h * g), ss[r][t] = sum of
// h^2 over columns 128t..128t+127.  One CTA per row, d/8 threads, 8 columns each.
struct EmbedParams {
  const int32_t* x;       // canvas [b][T]
  const uint16_t* embed;  // [V+1][d]
  const uint16_t* g;      // first RMSNorm gain [d]
  float* h;
  uint16_t* xn;
  uint16_t* xn_lo;        // bf16(h * g - xn), or null
  float* ss;
  int d, R, row0, T;
};

static __global__ void __launch_bounds__(1024) embed_kernel(const EmbedParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int seq = r / p.R, pos = p.row0 + r % p.R;
  const int tok = p.x[(long long)seq * p.T + pos];
  const int c0 = threadIdx.x * 8;
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
  if (p.xn_lo) *reinterpret_cast<uint4*>(p.xn_lo + (long long)r * p.d + c0) = *reinterpret_cast<const uint4*>(lv);
  // 16 threads cover one 128-column tile
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, s);
  if ((threadIdx.x & 15) == 0) p.ss[(long long)r * (p.d >> 7) + (c0 >> 7)] = sq;
}

// ------------------------------------------------------------------ selection
struct SelectRule {
  int policy;   // 0 threshold, 1 fixed-k, 2 factor, 3 budget
  float tau;
  int k;
  float factor;
};

// Select among the B positions of one sequence's block and commit.  Runs on
// a group of nthr threads (tid 0..nthr-1) that synchronise with sync();
// conf_s / arg_s / rank_s / eps_s in shared memory.  Writes x and the count
// (*count_out, by tid 0).
template <typename Sync>
__device__ __forceinline__ void select_commit_group(const float* conf_s, const int* arg_s, int* rank_s, float* eps_s,
                                                    int B, int32_t* xblk, int mask_id, const SelectRule rule,
                                                    int32_t* count_out, int* shared_best, int tid, int nthr,
                                                    Sync sync) {
  // eligibility and confidence rank (descending confidence, ties by position)
  for (int i = tid; i < B; i += nthr) {
    const bool e = xblk[i] == mask_id;
    int rank = -1;
    if (e) {
      rank = 0;
      const float ci = conf_s[i];
      for (int j = 0; j < B; ++j) {
        if (j == i || xblk[j] != mask_id) continue;
        const float cj = conf_s[j];
        rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
      }
    }
    rank_s[i] = rank;
  }
  if (tid == 0) *shared_best = 0;
  sync();
  int n_sel = 0;  // select ranks < n_sel
  if (rule.policy == 0) {
    // threshold: count qualifying positions
    for (int i = tid; i < B; i += nthr)
      if (rank_s[i] >= 0 && conf_s[i] >= rule.tau) atomicAdd(shared_best, 1);
    sync();
    const int nq = *shared_best;
    sync();
    for (int i = tid; i < B; i += nthr) {
      const int rk = rank_s[i];
      bool sel = false;
      if (rk >= 0) sel = (nq > 0) ? (conf_s[i] >= rule.tau) : (rk == 0);
      eps_s[i] = sel ? 1.0f : 0.0f;
    }
  } else {
    if (rule.policy == 1) {
      n_sel = rule.k;
    } else if (rule.policy == 4) {
      // scheduled: the MASK count spread over the k steps left (may be 0)
      for (int i = tid; i < B; i += nthr)
        if (rank_s[i] >= 0) atomicAdd(shared_best, 1);
      sync();
      n_sel = *shared_best / max(rule.k, 1);
    } else if (rule.policy == 2) {
      // factor: largest n with (n+1)(1 - c_(n)) < f, c_(n) = confidence of rank n-1
      for (int i = tid; i < B; i += nthr) {
        const int rk = rank_s[i];
        if (rk >= 0) {
          const float lhs = __fmul_rn((float)(rk + 2), __fsub_rn(1.0f, conf_s[i]));
          if (lhs < rule.factor) atomicMax(shared_best, rk + 1);
        }
      }
      sync();
      n_sel = max(*shared_best, 1);
    } else {
      // eq. 9 budget: sequential float32 prefix sum in rank order
      for (int i = tid; i < B; i += nthr)
        if (rank_s[i] >= 0) eps_s[rank_s[i]] = __fsub_rn(1.0f, conf_s[i]);
      sync();
      if (tid == 0) {
        int m = 0;
        for (int i = 0; i < B; ++i) m += rank_s[i] >= 0 ? 1 : 0;
        float total = 0.0f;
        int best = 0;
        for (int n = 1; n <= m; ++n) {
          const float e = eps_s[n - 1];
          total = __fadd_rn(total, e);
          if (__fadd_rn(total, e) < 1.0f) best = n;
        }
        *shared_best = best;
      }
      sync();
      n_sel = max(*shared_best, 1);
    }
    sync();
    for (int i = tid; i < B; i += nthr) {
      const int rk = rank_s[i];
      eps_s[i] = (rk >= 0 && rk < n_sel) ? 1.0f : 0.0f;
    }
  }
  sync();
  if (tid == 0) *shared_best = 0;
  sync();
  for (int i = tid; i < B; i += nthr) {
    if (eps_s[i] != 0.0f) {
      xblk[i] = arg_s[i];
      atomicAdd(shared_best, 1);
    }
  }
  sync();
  if (tid == 0) *count_out = *shared_best;
}

__device__ __forceinline__ void select_commit_cta(const float* conf_s, const int* arg_s, int* rank_s, float* eps_s,
                                                  int B, int32_t* xblk, int mask_id, const SelectRule rule,
                                                  int32_t* count_out, int* shared_best) {
  select_commit_group(conf_s, arg_s, rank_s, eps_s, B, xblk, mask_id, rule, count_out, shared_best, threadIdx.x,
                      blockDim.x, [] { __syncthreads(); });
}

// LM-head tile statistics -> (conf, arg) per block row, then select/commit.
// One CTA (256 threads) per block row merges that row's v_tiles statistics
// (fixed assignment and tree: deterministic); the last CTA of a sequence to
// finish runs the selection over the sequence's B rows.
struct MergeParams {
  const float* st_m;
  const float* st_s;
  const int* st_a;
  int v_tiles, n_rows;    // tiles, rows of the stat arrays (= b * B)
  int B, T, blk_start, mask_id;
  int32_t* x;             // canvas [b][T]
  float* conf;            // [b][B]
  int32_t* arg;           // [b][B]
  int32_t* count;         // [b]
  int* seq_done;          // [b] arrival counters, zero between launches
  SelectRule rule;
};

constexpr int kMaxBlock = 256;

struct MaxSumArg {
  float m, s;
  int a;
};

// (m1, s1, a1) + (m2, s2, a2): the larger maximum wins, sums rescaled to it,
// equal maxima keep the lower id.  The argument order fixes the rounding.
__device__ __forceinline__ MaxSumArg msa_merge(MaxSumArg x, MaxSumArg y) {
  const float M = fmaxf(x.m, y.m);
  const float sx = (x.m == -INFINITY) ? 0.0f : x.s * exp2f((x.m - M) * kLog2e);
  const float sy = (y.m == -INFINITY) ? 0.0f : y.s * exp2f((y.m - M) * kLog2e);
  MaxSumArg r;
  r.m = M;
  r.s = sx + sy;
  r.a = (y.m > x.m || (y.m == x.m && y.a < x.a)) ? y.a : x.a;
  return r;
}

static __global__ void __launch_bounds__(256) merge_select_kernel(const MergeParams p) {
  __shared__ MaxSumArg part[8];
  __shared__ float conf_s[kMaxBlock];
  __shared__ int arg_s[kMaxBlock];
  __shared__ int rank_s[kMaxBlock];
  __shared__ float eps_s[kMaxBlock];
  __shared__ int best;
  __shared__ int last;
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.x;              // seq * B + i
  const int seq = row / p.B;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  MaxSumArg acc{-INFINITY, 0.0f, 0x7fffffff};
  for (int t = threadIdx.x; t < p.v_tiles; t += 256) {
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
  __syncthreads();
  if (threadIdx.x == 0) {
    MaxSumArg r = part[0];
    for (int w = 1; w < 8; ++w) r = msa_merge(r, part[w]);
    p.conf[row] = 1.0f / r.s;
    p.arg[row] = r.a;
    __threadfence();
    const int old = atomicAdd(&p.seq_done[seq], 1);
    last = (old == p.B - 1);
    if (last) p.seq_done[seq] = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < p.B; i += 256) {
    conf_s[i] = __ldcg(&p.conf[(long long)seq * p.B + i]);
    arg_s[i] = __ldcg(&p.arg[(long long)seq * p.B + i]);
  }
  __syncthreads();
  select_commit_cta(conf_s, arg_s, rank_s, eps_s, p.B, p.x + (long long)seq * p.T + p.blk_start, p.mask_id,
                    p.rule, p.count + seq, &best);
}

// Standalone select/commit on given confidences (the K7 unit).
struct SelectParams {
  const float* conf;
  const int32_t* arg;
  int32_t* x;
  int32_t* count;
  int T, blk_start, B, mask_id;
  SelectRule rule;
};

static __global__ void __launch_bounds__(256) select_kernel(const SelectParams p) {
  __shared__ float conf_s[kMaxBlock];
  __shared__ int arg_s[kMaxBlock];
  __shared__ int rank_s[kMaxBlock];
  __shared__ float eps_s[kMaxBlock];
  __shared__ int best;
  const int seq = blockIdx.x;
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
    conf_s[i] = p.conf[(long long)seq * p.B + i];
    arg_s[i] = p.arg[(long long)seq * p.B + i];
  }
  __syncthreads();
  select_commit_cta(conf_s, arg_s, rank_s, eps_s, p.B, p.x + (long long)seq * p.T + p.blk_start, p.mask_id,
                    p.rule, p.count + seq, &best);
}

}  // namespace dllm
