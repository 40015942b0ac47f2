"""Model shapes and synthetic workloads of the cached masked-diffusion decoder.

Every model is a bidirectional (non-causal) LLaMA-style transformer as the
Fast-dLLM pages describe it (dian8dian "Fast-dLLM" summary, section on dLLM
mechanics; zhongzhuzhou.org reading notes, section 2, eq. 3): pre-norm blocks
``h += Attn(RMSNorm(h))`` and ``h += W_d(silu(W_g x) * W_u x)`` with
``x = RMSNorm(h)``, multi-head attention with scale 1/sqrt(head_dim), rotate-half
RoPE at absolute positions, no biases, untied embedding / LM head, and a MASK
token whose id equals ``vocab`` (the embedding therefore has ``vocab + 1`` rows
and the LM head ``vocab`` rows, so an argmax never yields MASK).

``lm_scale`` multiplies the standard deviation of the LM-head init.  Given an
RMS-normalised hidden row, the logits over a random N(0, 0.02*s) head are iid
Gaussian with sigma = 0.02 * s * sqrt(d_model); sigma = 12 puts the median
max-softmax confidence near 0.75-0.88 with ~40% of positions at >= 0.9 for every
vocabulary size used here.  The tiny model keeps its stated x8 (sigma = 2.56);
``tiny_spread`` is the same model at sigma = 10.
"""
from __future__ import annotations

import dataclasses
import math


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    rope_theta: float = 1e4
    norm_eps: float = 1e-5
    init_std: float = 0.02
    lm_scale: float = 1.0

    @property
    def mask_id(self) -> int:
        return self.vocab

    @property
    def lm_std(self) -> float:
        return self.init_std * self.lm_scale

    def n_params_layers(self) -> int:
        d, f = self.d_model, self.d_ffn
        return self.n_layers * (4 * d * d + 3 * d * f + 2 * d)

    def weight_bytes_step(self) -> int:
        """bf16 bytes of every matrix one denoise step streams (layers + LM head)."""
        d, f = self.d_model, self.d_ffn
        per_layer = 4 * d * d + 3 * d * f
        return 2 * (self.n_layers * per_layer + self.vocab * d)

    def kv_bytes(self, T: int, batch: int = 1) -> int:
        """bf16 bytes of the K/V cache of ``batch`` sequences of length T."""
        return 2 * 2 * self.n_layers * batch * T * self.d_model


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    batch: int
    prompt_len: int
    gen_len: int
    block: int
    tau: float = 0.9
    seed: int = 0

    @property
    def T(self) -> int:
        return self.prompt_len + self.gen_len


def _sigma_scale(sigma: float, d: int, std: float = 0.02) -> float:
    return sigma / (std * math.sqrt(d))


TINY = ModelConfig("tiny", 2, 256, 4, 64, 688, 1024, lm_scale=8.0)
TINY_SPREAD = dataclasses.replace(TINY, name="tiny_spread", lm_scale=31.25)
M1B = ModelConfig("1b", 16, 2048, 16, 128, 5504, 32000, lm_scale=13.25)
M8B = ModelConfig("8b", 32, 4096, 32, 128, 12288, 126464, lm_scale=9.375)

MODELS = {m.name: m for m in (TINY, TINY_SPREAD, M1B, M8B)}

WORKLOADS = {
    "tiny": Workload("tiny", TINY, 1, 32, 64, 16),
    "tiny_spread": Workload("tiny_spread", TINY_SPREAD, 1, 32, 64, 16),
    "1b": Workload("1b", M1B, 1, 256, 128, 32),
    "8b": Workload("8b", M8B, 1, 512, 256, 32),
    "8b_long": Workload("8b_long", M8B, 1, 1024, 1024, 32),
    "8b_batch": Workload("8b_batch", M8B, 1, 128, 128, 32),
}
# Denoise steps and refreshes per generation that the GPU path takes on a
# workload's seeded inputs (batch as listed, DualCache, the workload's tau,
# bidirectional mask, split precision): measured on GB300, deterministic for
# the seed.  The CPU oracle's timed sample is extrapolated with these counts,
# so that both arms of the bench describe the same generation.
STEPS_PER_GENERATION = {
    "8b": (117, 8),
    "1b": (59, 4),
}

BATCH_SWEEP = (1, 2, 4, 8, 16, 32, 64)
TAU_SWEEP = (0.7, 0.8, 0.9, 0.95)
