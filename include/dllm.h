/*
 * dllm.h - C ABI of the GB300 (sm_103a) block-cached, confidence-threshold
 * masked-diffusion decoder.
 *
 * The method (Fast-dLLM, as described in the zhongzhuzhou.org reading notes,
 * sections 3-6, and the dian8dian summary): the answer of length gen_len is
 * split into blocks of B positions decoded left to right (Algorithm 1).  While
 * the current block still holds MASK, one denoise step runs a bidirectional
 * transformer forward over the recomputed rows only - the current block
 * (DualCache), the block and the suffix (PrefixCache) or every position (no
 * cache) - reading cached K/V for the other positions; it takes, for every
 * masked position of the block, the largest softmax probability c_i and the
 * argmax token y_i over the vocabulary, and commits every position with
 * c_i >= tau, or only the single most confident one if none qualifies
 * (Algorithm 2).  A committed token is never changed again.  At each block
 * boundary a full-sequence forward rewrites every cached K/V in place.
 *
 * Conventions
 *  - Every call returns a dllm_status (dllm_denoise_step returns a count, or a
 *    negative status).  On failure dllm_last_error() holds a message (per
 *    thread) and no state has changed unless the text says otherwise.
 *  - Host pointers are owned by the caller and only read/written during the
 *    call.  Device memory of models and states is owned by the library and
 *    freed by dllm_free_model / dllm_free_state.
 *  - A dllm_state is used by one host thread at a time.  Calls are
 *    synchronous with respect to the host outputs they return.
 *  - Token ids are int32 in [0, vocab); the MASK id is `vocab`.
 *  - The dllm_op_* calls take device pointers, run on the given CUDA stream
 *    (NULL = legacy default stream) and return after the launch (asynchronous).
 */
#ifndef DLLM_H
#define DLLM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dllm_status {
    DLLM_OK = 0,
    DLLM_EINVAL = 1,    /* bad argument; nothing was changed */
    DLLM_ENOMEM = 2,    /* device or host allocation failed */
    DLLM_ECUDA = 3,     /* a CUDA runtime/driver call failed */
    DLLM_EIO = 4,       /* weight file missing, short or malformed */
    DLLM_ESTATE = 5,    /* a step committed nothing while MASK remained, or the
                           call does not fit the state (e.g. wrong block) */
    DLLM_ETIMEOUT = 6,  /* a kernel gave up a bounded wait; outputs are invalid */
    DLLM_ECANCELLED = 7 /* dllm_run stopped because its run hook returned nonzero */
} dllm_status;

typedef enum dllm_cache_mode {
    DLLM_CACHE_NONE = 0,    /* every step recomputes all T positions */
    DLLM_CACHE_PREFIX = 1,  /* recompute the current block and the suffix */
    DLLM_CACHE_DUAL = 2     /* recompute only the current block */
} dllm_cache_mode;

typedef enum dllm_sel_policy {
    DLLM_SEL_THRESHOLD = 0, /* Algorithm 2: c >= tau, else the single best */
    DLLM_SEL_FIXED_K = 1,   /* the k most confident (min(k, remaining)) */
    DLLM_SEL_FACTOR = 2,    /* Algorithm 3 / eq. 13: largest n with (n+1)(1-c_(n)) < f */
    DLLM_SEL_BUDGET = 3,    /* eq. 9: largest prefix with sum eps + max eps < 1 */
    DLLM_SEL_SCHEDULE = 4   /* page 1's LLaDA remasking schedule: with k steps left in the
                               block, the n_keep = (MASK count) / k most confident (n_keep
                               may be 0); dllm_run counts k down from the given k per block */
} dllm_sel_policy;

/* Selection rule.  Ties in confidence go to the lowest position, ties in the
 * argmax to the lowest token id; every comparison is made in float32 on the
 * float32 confidence.  Only MASK positions of the current block are eligible. */
typedef struct dllm_select {
    int32_t policy;   /* dllm_sel_policy */
    float tau;        /* THRESHOLD: threshold (> 1 gives one token per step) */
    int32_t k;        /* FIXED_K: tokens per step, >= 1 */
    float factor;     /* FACTOR: f > 0 */
} dllm_select;

/* Model shape (LLaMA-style, non-causal, MHA with n_heads * head_dim = d_model,
 * rotate-half RoPE, RMSNorm, SwiGLU FFN, untied embedding [vocab+1][d] and
 * LM head [vocab][d]).  head_dim must be 64 or 128; d_model a multiple of 128. */
typedef struct dllm_config {
    int32_t n_layers, d_model, n_heads, head_dim, d_ffn, vocab;
    float rope_theta, norm_eps;
} dllm_config;

/* Logical weight tensors, row-major [out][in] bf16 (uint16 bit patterns). */
typedef enum dllm_tensor {
    DLLM_T_EMBED = 1,       /* [vocab+1][d]  (row `vocab` is MASK)   */
    DLLM_T_ATTN_NORM = 2,   /* [d]    per layer                        */
    DLLM_T_WQ = 3,          /* [d][d] per layer, out = head*head_dim+j */
    DLLM_T_WK = 4,
    DLLM_T_WV = 5,
    DLLM_T_WO = 6,          /* [d][d] per layer                        */
    DLLM_T_FFN_NORM = 7,    /* [d]    per layer                        */
    DLLM_T_WG = 8,          /* [d_ffn][d] per layer                    */
    DLLM_T_WU = 9,          /* [d_ffn][d] per layer                    */
    DLLM_T_WD = 10,         /* [d][d_ffn] per layer                    */
    DLLM_T_FINAL_NORM = 11, /* [d]                                     */
    DLLM_T_LM_HEAD = 12     /* [vocab][d]                              */
} dllm_tensor;

/* Timings and counts of one dllm_run / dllm_generate (eq. 15 of the notes:
 * T_fast ~ S * C_active + R + T_selection; selection runs inside the step). */
typedef struct dllm_stats {
    double wall_ms;       /* whole call, host clock                             */
    double refresh_ms;    /* R: prefill + refreshes (CUDA events), the fused
                             refresh-and-step forwards included                 */
    double step_ms;       /* the other denoise steps (CUDA events)               */
    int32_t steps;        /* S: denoise steps run, fused ones included           */
    int32_t refreshes;    /* full-sequence forwards (prefill included)           */
    int32_t blocks;
    int32_t max_steps_per_block;
    int64_t committed;    /* tokens committed over all sequences                 */
    double tau_bar;       /* committed / sum over sequences of active steps      */
    int64_t kernel_launches; /* kernels this call launched                       */
    int32_t fused_steps;  /* steps run as the forward of the refresh before them
                             (counted in steps and in refreshes; their time is in
                             refresh_ms): C_active = step_ms / (steps - fused)   */
    int32_t reserved;
} dllm_stats;

typedef struct dllm_model dllm_model;
typedef struct dllm_state dllm_state;

/* ------------------------------------------------------------------ model */

/* Allocate a model's device weights (uninitialised) on the current device.
 * Fill every tensor with dllm_model_set_tensor before use. */
dllm_status dllm_model_create(const dllm_config* cfg, dllm_model** out);

/* Copy one logical tensor (count bf16 values, row-major [out][in]) into the
 * model's device layout.  src is a host pointer (src_on_device = 0) or a
 * device pointer (1).  count must equal the tensor's element count. */
dllm_status dllm_model_set_tensor(dllm_model* m, int32_t tensor, int32_t layer,
                                  const uint16_t* src, int64_t count, int32_t src_on_device);

/* Read a weight file and upload it: the model-loading call the decoder's
 * interface starts from (a trained model's weights in the pages' setting;
 * here seeded random-init weights of the same shapes).  Format: 8-byte magic
 * "DLLMW001", int32 n_layers, d_model,
 * n_heads, head_dim, d_ffn, vocab, float32 rope_theta, norm_eps, then every
 * tensor's bf16 bits: embed; per layer attn_norm wq wk wv wo ffn_norm wg wu wd;
 * final_norm; lm_head) and upload it.  DLLM_EIO on a short/malformed file. */
dllm_status dllm_load(const char* path, dllm_model** out);

dllm_status dllm_model_config(const dllm_model* m, dllm_config* cfg);
void dllm_free_model(dllm_model* m);

/* ------------------------------------------------------------------ state */

/* Create the decoding state of b sequences: canvas x = prompt ++ MASK*gen_len
 * (Algorithm 1 of the Fast-dLLM reading notes, section 3, step 1: append
 * gen_len MASK positions to the prompt; the tutorial's sampler starts from the
 * same all-MASK answer), K/V cache [layer][K|V][b][head][T][head_dim] bf16 with
 * T = P + gen_len, activations and workspaces.  prompts: host [b][P] int32, or
 * NULL to leave the prompt part for dllm_state_set_prompts_device.
 * gen_len % block == 0 and 1 <= block <= 256 are required.  cuda_stream is a
 * cudaStream_t (NULL = create a private stream).  Nothing runs on the GPU. */
dllm_status dllm_state_create(dllm_model* m, const int32_t* prompts, int32_t b, int32_t P,
                              int32_t gen_len, int32_t block, void* cuda_stream,
                              dllm_state** out);

/* Reset the canvas to prompt ++ MASK (prompts: host [b][P], or NULL to keep
 * the current prompt part) and forget the cache contents and counters. */
dllm_status dllm_state_reset(dllm_state* s, const int32_t* prompts);

/* Copy prompts already on the device ([b][P] int32) into the canvas and reset
 * the answer part to MASK (stream-ordered, no host synchronisation). */
dllm_status dllm_state_set_prompts_device(dllm_state* s, const int32_t* prompts_dev);

void dllm_free_state(dllm_state* s);

/* Full-sequence forward over all T positions of the current canvas; writes
 * every layer's K and V for every position into the cache in place (Algorithm
 * 1, steps 2 and 11).  Commits nothing; skips the last layer's attention/FFN
 * and the LM head, which K/V do not need. */
dllm_status dllm_prefill_refresh(dllm_state* s);

/* One denoise step of block block_idx with the threshold rule (Algorithm 2)
 * and the given cache mode.  committed_per_seq: host [b] or NULL.  Returns the
 * total number of tokens committed (>= 0), or -status on error.  A sequence
 * whose block has no MASK left commits 0.  block_idx must be in
 * [0, gen_len/block).  The cached modes read whatever the cache holds: call
 * dllm_prefill_refresh first. */
int32_t dllm_denoise_step(dllm_state* s, int32_t block_idx, float tau, int32_t cache_mode,
                          int32_t* committed_per_seq);

/* Same with any selection rule. */
dllm_status dllm_denoise_step_ex(dllm_state* s, int32_t block_idx, const dllm_select* sel,
                                 int32_t cache_mode, int32_t* committed_per_seq);

/* Algorithm 1 on the state's canvas: prefill refresh (cached modes), then for
 * each block, denoise steps until it has no MASK, then a refresh before the
 * next block (cached modes).  Tokens stay on the device (read them with
 * dllm_read_state).  refresh_interval > 0 also refreshes after every
 * refresh_interval steps inside a block (0 = only at block boundaries).
 * A refresh and the step after it run as one full forward over all T rows:
 * it rewrites every layer's K/V from the canvas, as the refresh does, and its
 * block rows are the step's, which after a refresh reads exactly those K/V
 * (stats->fused_steps counts them).  Under the block-causal mask this covers
 * the prefill and a refresh interval's refreshes, and in DualCache runs each
 * block-boundary commit forward (block j's K/V from the final canvas) runs in
 * one launch with block j+1's first step, over both blocks' rows.  The run
 * hook still sees the refresh (or commit-forward) event, then the step event.
 * stats may be NULL. */
dllm_status dllm_run(dllm_state* s, const dllm_select* sel, int32_t cache_mode,
                     int32_t refresh_interval, dllm_stats* stats);

/* Observer of dllm_run (and of nothing else): called on the calling thread
 * after each event of the loop has completed on the GPU, with the event kind,
 * the block index j and the step's index inside the block (for a refresh: the
 * number of steps the block had taken).  Events: DLLM_EVENT_REFRESH after the
 * prefill and every refresh (block boundary, or the refresh interval inside a
 * block), DLLM_EVENT_STEP after every denoise step, DLLM_EVENT_COMMIT_FORWARD
 * after the forward over a finished block that replaces the block-boundary
 * refresh under the block-causal mask.  A refresh (or commit forward) that
 * runs in one forward with the step after it is reported right before that
 * step's event, once both are done: the canvas then already holds the step's
 * commits.  Inside the hook the state may be read (dllm_read_state,
 * dllm_read_hidden, dllm_read_kv) but not changed.  A nonzero return stops
 * the run: dllm_run returns DLLM_ECANCELLED, with the canvas as the last
 * completed forward left it.  Use: stream committed tokens to a caller, or
 * follow the loop's decisions step by step. */
typedef enum dllm_event { DLLM_EVENT_REFRESH = 0, DLLM_EVENT_STEP = 1, DLLM_EVENT_COMMIT_FORWARD = 2 } dllm_event;
typedef int32_t (*dllm_run_hook)(void* user, int32_t event, int32_t block_idx, int32_t step_in_block);

/* Install (or with hook NULL remove) the state's run hook; user is passed back
 * unchanged.  It stays installed until changed or the state is freed. */
dllm_status dllm_state_set_run_hook(dllm_state* s, dllm_run_hook hook, void* user);

/* End-to-end call: prompts (host [b][P]) in, answers (host [b][gen_len]) out.
 * Creates a state on a private stream, runs Algorithm 1 with the threshold
 * rule, copies the answer back and frees the state. */
dllm_status dllm_generate(dllm_model* m, const int32_t* prompts, int32_t b, int32_t P,
                          int32_t gen_len, int32_t block, float tau, int32_t cache_mode,
                          int32_t* out_tokens, dllm_stats* stats);

/* Copy state to the host: tokens [b][T] (the whole canvas; Algorithm 1 of the
 * Fast-dLLM reading notes, section 3, returns its answer part), and the last
 * step's conf [b][block] (float32 max-softmax c_i) and arg [b][block] (argmax
 * y_i), the candidates and confidences of Algorithm 2 (section 4, steps 1-2).
 * Any pointer may be NULL. */
dllm_status dllm_read_state(const dllm_state* s, int32_t* tokens, float* conf, int32_t* arg);

/* The last denoise step's residual stream after the last layer for the block
 * rows, host float32 [b][block][d_model]. */
dllm_status dllm_read_hidden(const dllm_state* s, float* h);

/* Copy the cached K and V of one layer as float32, host [b][n_heads][T][head_dim] each
 * (hi + lo in split precision). */
dllm_status dllm_read_kv(const dllm_state* s, int32_t layer, float* k, float* v);

/* Precision of the activations fed to the tensor cores.  DLLM_PREC_SPLIT
 * (default) carries every GEMM input as a pair of bf16 arrays hi + lo with
 * lo = bf16(x - hi) (about 16 mantissa bits; the weights are read once, the
 * MMA is twice as wide).  DLLM_PREC_BF16 rounds activations to bf16 (half the
 * tensor work: for the compute-bound batch regime).  In split precision the
 * K/V cache, q and the attention probabilities are hi/lo pairs as well (the
 * cache holds both halves: twice the K/V bytes); in bf16 precision they are
 * bf16.  Accumulation is float32 in both.  Change the precision only before a
 * refresh: the cache's low halves are written only in split precision. */
typedef enum dllm_precision { DLLM_PREC_SPLIT = 0, DLLM_PREC_BF16 = 1 } dllm_precision;
dllm_status dllm_state_set_precision(dllm_state* s, int32_t mode);

/* DualCache steps with at most 128 activation rows (b * block <= 128, block
 * <= 32) run by default as one persistent cooperative launch: one CTA per SM
 * walks through every phase of the step (embedding, each layer's projections
 * and attention, LM head, merge and selection), ordered by dataflow flags (a
 * consumer waits only for the row tiles or heads it reads, no grid-wide
 * barrier), and streams the next phase's weights while a phase finishes.
 * enable 0 selects one launch per kernel instead (same arithmetic except the
 * attention key split; tracing always uses it). */
dllm_status dllm_state_set_persistent(dllm_state* s, int32_t enable);

/* dllm_run's fused forwards (on by default): a refresh and the step after it
 * run as one forward, and under the block-causal mask a DualCache run's
 * commit forward shares a launch with the next block's first step (see
 * dllm_run).  enable 0 runs every refresh and commit forward on its own, then
 * the step, as Algorithm 1 lists them; the trajectory is the same up to the
 * kernels' rounding. */
dllm_status dllm_state_set_fused_refresh(dllm_state* s, int32_t enable);

/* Run-ahead in dllm_run (enable 1, the default): within a block, the next
 * DualCache step that runs as one persistent launch is enqueued before the
 * current step's commit counts are read back, so the GPU does not wait for
 * the host between steps (Algorithm 1's inner loop, section 3 of the
 * Fast-dLLM reading notes, decides whether the block still holds a MASK only
 * after each step).  When the current step commits the block's last MASK,
 * the step launched ahead finds none at its start and ends without writing
 * anything; it is counted in kernel_launches, not in steps.  Tokens, steps
 * and refreshes are the same as with enable 0.  Run-ahead is off while a
 * run hook, per-kernel timing, the step timeline or the trace is set, and
 * for PrefixCache and no-cache runs, refresh-interval steps and steps that
 * do not fit one persistent launch. */
dllm_status dllm_state_set_run_ahead(dllm_state* s, int32_t enable);

/* Attention mask.  DLLM_MASK_BIDIRECTIONAL (default): every position sees
 * every position, the Fast-dLLM setting, in which the cached prefix and
 * suffix go stale and a block-boundary refresh recomputes them.
 * DLLM_MASK_BLOCK_CAUSAL: a prompt position sees the prompt, a position of
 * answer block j the prompt and blocks 0..j (block diffusion, BD3-LM style,
 * which the tutorial's section on caches and the dian8dian summary name as
 * the exact-cache alternative).  Nothing then attends to a later block, the
 * cache never goes stale, PrefixCache and DualCache compute the same as no
 * cache, and dllm_run replaces each block-boundary refresh by one forward
 * over the finished block's rows that caches their K/V.  Set before
 * dllm_prefill_refresh.  DLLM_EINVAL for another value. */
typedef enum dllm_mask { DLLM_MASK_BIDIRECTIONAL = 0, DLLM_MASK_BLOCK_CAUSAL = 1 } dllm_mask;
dllm_status dllm_state_set_mask(dllm_state* s, int32_t mask);

/* Diagnostics of the persistent step: with enable 1 the next persistent steps
 * record, per CTA and phase, 10 %globaltimer nanosecond stamps (uint64
 * [ctas][phases][10]): 0 the CTA's workers finished the phase, 1 its TMA
 * producer issued the phase's first activation tile (entry [cta][0][1] is the
 * kernel start), 2 its MMA issuer finished the phase, 3 the producer issued
 * the phase's last tile, 4 the workers started the phase, 5 they got its
 * first accumulator, 6 they were through their first segment, 7 they started
 * their last stream-K fix-up as the last contributor, 8 they had summed its
 * partials, 9 they published their last unit (row tile) of the phase; for
 * attention phases 5-9 are: first item's inputs ready, first item done, its
 * keys done, its split partial stored and counted, last head published; 0
 * where an event did not occur.  dllm_read_step_timeline copies the last step's
 * record. */
dllm_status dllm_state_set_step_timeline(dllm_state* s, int32_t enable);
dllm_status dllm_read_step_timeline(const dllm_state* s, uint64_t* out, int64_t capacity, int32_t* ctas,
                                    int32_t* phases);

/* Record the residual stream after the embedding and after every layer on the
 * next steps (1) or stop (0).  dllm_read_trace copies the last step's record,
 * host float32 [n_layers+1][rows][d_model], rows = b * rows_per_seq as
 * returned.  Tracing adds copies between layers: not for timing. */
dllm_status dllm_state_set_trace(dllm_state* s, int32_t enable);
dllm_status dllm_read_trace(const dllm_state* s, float* out, int64_t capacity_floats,
                            int32_t* rows_per_seq, int32_t* first_pos);

/* Accumulate per-kernel-class device time of the next calls with CUDA events
 * (enable 1), or stop (0).  dllm_kernel_times returns, per class, the summed
 * milliseconds, launch counts and algorithmic bytes (weights, K/V and
 * activations each counted once).  Classes of a denoise step: 0 embed,
 * 1 qkv_gemm, 2 attention, 3 o_gemm, 4 gateup_gemm, 5 down_gemm,
 * 6 lm_head_gemm, 7 merge_select; a refresh's launches use 8 + the same index;
 * 14 is the persistent step kernel.  16 classes in all.  The events serialise the kernels: not for the headline
 * time. */
dllm_status dllm_state_set_kernel_timing(dllm_state* s, int32_t enable);
dllm_status dllm_kernel_times(const dllm_state* s, double* ms, int64_t* launches,
                              double* bytes, int32_t n_classes);

/* ------------------------------------------------------------------ kernels */

/* Y[N][M] (float32) = X[N][K] * W[M][K]^T on the tensor cores (tcgen05, TMA,
 * stream-K split with a deterministic fix-up).  W, X bf16 row-major, 16-byte
 * aligned, K % 8 == 0.  X_lo (nullable) is a second bf16 array added to X
 * (the hi/lo activation pair).  Uses a library-owned workspace allocated on
 * first use. */
dllm_status dllm_op_gemm(const uint16_t* W, const uint16_t* X, const uint16_t* X_lo, float* Y,
                         int32_t M, int32_t N, int32_t K, void* cuda_stream);

/* dllm_op_gemm with a per-CTA timeline for diagnostics: trace (device,
 * uint64 [grid][8], grid <= the SM count, returned in *grid_out) receives per
 * CTA {SM id, start, first operand tile landed, last MMA issued, epilogue done,
 * end} in %globaltimer nanoseconds (entries 6-7 unused).  trace may be NULL. */
dllm_status dllm_op_gemm_trace(const uint16_t* W, const uint16_t* X, const uint16_t* X_lo, float* Y,
                               int32_t M, int32_t N, int32_t K, uint64_t* trace, int32_t* grid_out,
                               void* cuda_stream);

/* Non-causal attention, eq. 3: for every sequence s, head h and query row i,
 * out[s*R+i][h*hd..] = softmax(q k^T / sqrt(hd)) v over the T keys of
 * k_cache/v_cache [b][H][T][hd].  q: [b*R][H][hd] bf16, out [b*R][H*hd] bf16.
 * hd in {64, 128}.  Splits the keys across CTAs and merges the partial
 * softmax states deterministically (library-owned workspace). */
dllm_status dllm_op_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                              uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R,
                              int32_t T, void* cuda_stream);

/* The same attention (eq. 3 of the Fast-dLLM reading notes, section 2; same
 * arguments, layouts and output as dllm_op_attention) on the tensor cores:
 * one CTA per (128-query tile, key split, head, sequence) runs S = q K^T and
 * O = P V as tcgen05.mma with S and O in tensor memory.  The keys are split
 * (at most 8 ways, 64-key granularity) when the query tiles alone would fill
 * the GPU's SMs unevenly; the last split of a query tile to finish merges the
 * partial softmax states in split order (deterministic), in a library-owned
 * workspace grown on first use.  This is the kernel the library uses for 65
 * or more query rows per sequence (the refresh's full forward, PrefixCache
 * and no-cache steps); block queries use the key-split kernel.  q, k_cache,
 * v_cache and out must be 16-byte aligned.  Results agree with
 * dllm_op_attention to bf16 rounding of the probabilities and the output,
 * not bit for bit. */
dllm_status dllm_op_attention_tc(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                 uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R,
                                 int32_t T, void* cuda_stream);

/* dllm_op_attention_tc with the number of key splits chosen by the caller:
 * splits = 0 takes the library's plan (as dllm_op_attention_tc), 1..8 cuts
 * the keys into that many ranges of equal 64-key multiples (fewer when T is
 * short: ranges past T are dropped).  Other values: DLLM_EINVAL. */
dllm_status dllm_op_attention_tc_ex(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                    uint16_t* out, int32_t b, int32_t H, int32_t hd, int32_t R,
                                    int32_t T, int32_t splits, void* cuda_stream);

/* dllm_op_attention with no allocation of any kind.  The pages have no
 * counterpart to this entry point: it computes the same attention as
 * dllm_op_attention, with the same arguments, layouts and output, and is
 * bit-identical to it for every shape it accepts.  What differs is where the
 * scratch lives.  dllm_op_attention grows a library-owned workspace with
 * cudaMalloc + cudaMemset the first time a shape needs more; this variant uses
 * a fixed scratch in static device storage of the library (key-split
 * partials: 1 Mi floats = 4 MiB; merge counters: 4096; every device that
 * loads the library holds it until the process exits) and never calls
 * cudaMalloc, cudaFree or an allocating library.  It serves callers that must
 * not allocate device memory at call time: a caller whose device memory is
 * fully reserved up front (weights and K/V pools sized to the card), or one
 * that issues work where an allocation, or the device-wide synchronisation a
 * cudaMalloc may imply, is not allowed.
 *  - Set-up: the first call on each device looks up the scratch's device
 *    address (cudaGetSymbolAddress with that device current) and the driver's
 *    tensor-map entry point; make that first call before any stream capture.
 *  - Limit: b*H*ceil(R/QT) merge works and, when the keys are split,
 *    works*splits*QT*(hd+2) floats (QT = 32 for R <= 32, else 64; splits as
 *    dllm_op_attention plans them for this GPU).  A call over the limit
 *    returns DLLM_EINVAL, launches nothing and names the limit in
 *    dllm_last_error(); use dllm_op_attention for it.  The 8B DualCache block
 *    (b=1, H=32, hd=128, R=32, T=768) fits.
 *  - Zero state: each call clears the merge counters it uses (a
 *    cudaMemsetAsync on the caller's stream) before its launch, so a call
 *    after one that gave up a bounded wait starts clean.
 *  - Errors: a launch that gives up a bounded wait sets the scratch's error
 *    word; dllm_op_check reports it (DLLM_ETIMEOUT) and clears it.
 *  - Concurrency: all calls on a device share the one scratch.  Calls ordered
 *    on one stream are safe; calls that may overlap (different streams, or
 *    different host threads without ordering) race on the scratch and give
 *    wrong results.
 *  - Asynchronous like dllm_op_attention: returns after the launch. */
dllm_status dllm_op_attention_noalloc(const uint16_t* q, const uint16_t* k_cache,
                                      const uint16_t* v_cache, uint16_t* out, int32_t b,
                                      int32_t H, int32_t hd, int32_t R, int32_t T,
                                      void* cuda_stream);

/* Synchronise cuda_stream, then report whether any kernel launched by the
 * dllm_op_* calls on the current device (the no-alloc attention included)
 * gave up a bounded wait since the last check: DLLM_ETIMEOUT with the wait's
 * site code in *site (nullable), else DLLM_OK with *site = 0.  Clears the
 * error words it read.  Outputs of a call that timed out are invalid.
 * Allocates nothing. */
dllm_status dllm_op_check(int32_t* site, void* cuda_stream);

/* Failure detection without a fault: one GPU thread waits, with the same
 * bounded dataflow wait the persistent step uses between its phases, until
 * the device int32 *flag reaches need or limit_us microseconds (1 ..
 * 2,000,000) have passed.  Synchronous; returns DLLM_OK if the flag was
 * reached and DLLM_ETIMEOUT if the wait gave up (through dllm_op_check, which
 * also clears the error word, so the next call starts clean).  With a flag
 * that nothing raises it exercises the give-up path: error word set, the
 * kernel returns, the context stays usable. */
dllm_status dllm_op_wait_probe(const int32_t* flag, int32_t need, int32_t limit_us, void* cuda_stream);

/* The selection/commit kernel alone: given conf [b][B] float32 and arg [b][B]
 * int32 (device), select on the MASK positions x[s][blk_start .. +B) of the
 * canvas x [b][T] (device int32), write the chosen arg ids into x and the
 * per-sequence counts into count [b] (device). */
dllm_status dllm_op_select_commit(const float* conf, const int32_t* arg, int32_t* x,
                                  int32_t b, int32_t T, int32_t blk_start, int32_t B,
                                  int32_t mask_id, const dllm_select* sel, int32_t* count,
                                  void* cuda_stream);

/* Cache staleness diagnostics for block block_idx of the current canvas (the
 * Fast-dLLM notes, section 14, Algorithm 4 steps 4-5: compare fresh and
 * cached representations and predictions at the positions about to be
 * committed; the notes' section 3 on what DualCache freezes).  Without
 * changing the canvas or the cache's prefix/suffix rows it runs a full
 * forward over all T positions of the current canvas into a scratch K/V
 * ("fresh") and the block forward twice, on the cache and on the fresh K/V,
 * and returns (host outputs):
 *   k_cos[l], v_cos[l]  float32 [n_layers]: the mean over sequences, heads
 *                       and every position outside the block of the cosine
 *                       between the cached and the fresh K (V) row;
 *   agree               the fraction of the block's MASK positions whose
 *                       argmax is the same from both;
 *   max_dconf           the largest |max-prob(cached) - max-prob(fresh)| there.
 * The block's own K/V rows in the cache are rewritten with the current
 * canvas's (as the next step would).  Allocates a second K/V of the cache's
 * size on first use.  DLLM_EINVAL for a bad block or NULL output. */
dllm_status dllm_staleness(dllm_state* s, int32_t block_idx, float* k_cos, float* v_cos, float* agree,
                           float* max_dconf);

/* ------------------------------------------------------------------ misc */

const char* dllm_last_error(void);
const char* dllm_status_string(int32_t status);
/* Library version as major*10000 + minor*100 + patch. */
int32_t dllm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DLLM_H */
