"""Analytic step-time bounds (the teaching roofline of the dLLM speed tutorial).

tianyi-zhang-02.github.io "dLLM: decoding steps, cache and real speed",
section "a hand-computed account (teaching model)": a forward over n positions
costs at least ``max(W_bytes / BW, n * 2N / FLOPS)``; reading the weights
dominates below the crossover n* = (W_bytes / BW) / (2N / FLOPS).  The same
formula restated with GB300's measured peaks gives the per-step lower bound the
bench reports beside its measured step time.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class Roofline:
    weight_bytes: float       # bytes streamed per forward
    flops_per_position: float  # 2N for an N-parameter model
    bw_bytes_s: float
    flops_s: float

    @property
    def weight_ms(self) -> float:
        return self.weight_bytes / self.bw_bytes_s * 1e3

    @property
    def position_ms(self) -> float:
        return self.flops_per_position / self.flops_s * 1e3

    def step_ms(self, n: float) -> float:
        return max(self.weight_ms, n * self.position_ms)

    @property
    def crossover(self) -> float:
        return self.weight_ms / self.position_ms


def teaching_h100() -> Roofline:
    """The tutorial's numbers: 7B bf16 (1.4e10 B, 2N = 1.4e10 flop), H100 SXM5
    3.352 TB/s and 989.4 dense bf16 TFLOPS."""
    return Roofline(1.4e10, 1.4e10, 3.352e12, 989.4e12)


def ar_tokens_s(r: Roofline, batch: int) -> float:
    """Autoregressive decode at concurrency b: b tokens per step of b positions."""
    return batch / r.step_ms(batch) * 1e3


def diffusion_tokens_s(r: Roofline, batch: int, block: int, tau_bar: float) -> float:
    """Block diffusion at concurrency b: tau_bar tokens per sequence per step of b*block positions."""
    return tau_bar * batch / r.step_ms(block * batch) * 1e3


def dual_step_bytes(weight_bytes: float, kv_bytes: float) -> float:
    """Algorithmic bytes of one DualCache step: every weight once plus the K/V cache once."""
    return weight_bytes + kv_bytes
