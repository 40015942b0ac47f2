/*
 * dllm_synth.h - seeded synthetic inputs on the device (libdllm_synth.so).
 *
 * Not part of the decoding method: random-init weights and uniform prompt ids
 * for benchmarks and tests, bit-identical to the numpy generator of
 * cached_masked_decoding_gb300/synth.py.  Counter-based SplitMix64 (Steele,
 * Lea & Flood, OOPSLA 2014): word(i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15).
 *
 * All functions enqueue one kernel on cuda_stream (NULL = legacy default
 * stream), return the cudaError_t of the launch as int (0 = success) and take
 * device pointers.
 */
#ifndef DLLM_SYNTH_H
#define DLLM_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dst[i] = bf16_rne(float32(z_i) * c + offset), i < count, where z_i is the
 * Irwin-Hall sum of the four 16-bit fields of word(first + i) minus 131070.
 * c = float32(std * sqrt(3) / 65536) is computed by the caller. */
int dllm_synth_fill_normal_bf16(uint16_t* dst, int64_t count, uint64_t key, float c, float offset,
                                int64_t first, void* cuda_stream);

/* dst[i] = value for i < count. */
int dllm_synth_fill_const_bf16(uint16_t* dst, int64_t count, uint16_t value, void* cuda_stream);

/* dst[i] = ((word(first + i) >> 32) * vocab) >> 32, uniform ids in [0, vocab). */
int dllm_synth_fill_ids(int32_t* dst, int64_t count, uint64_t key, int32_t vocab, int64_t first,
                        void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* DLLM_SYNTH_H */
