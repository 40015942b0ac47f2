"""Oracle forward pass of the bidirectional LLaMA-style denoiser (float64, numpy).

TEST INFRASTRUCTURE ONLY (see package header).

What it computes, and the passage each step follows:

* the network is decoder-only with non-causal attention (dian8dian "Fast-dLLM"
  summary, section "dLLM mechanics": LLaDA-style decoder-only, non-causal);
  every position attends to every position (zhongzhuzhou.org notes, section 2,
  eq. 3: Attn(Q,K,V) = softmax(Q K^T / sqrt(d)) V, with d read as the head
  dimension);
* the block pieces follow the stated LLaMA-style shape: RMSNorm pre-norm,
  rotate-half RoPE at absolute positions, SwiGLU FFN W_d(silu(W_g x) * W_u x),
  no biases; the confidence of a position is the largest softmax probability
  over the vocabulary and the candidate the argmax (notes, section 4,
  Algorithm 2, steps 1-2);
* a forward over a subset of rows reads the K/V of the other positions from a
  cache (notes, section 3, Algorithm 1, steps 5-7: PrefixCache recomputes the
  current block and the suffix, DualCache only the current block; the query
  reads freshly computed and cached K/V together).

Pins (tests/test_oracle_pins.py): RMSNorm scale invariance and unit RMS; RoPE
identity at position 0, a hand-rotated vector, norm preservation and the
relative-position property; attention with identical keys = mean of V, a
two-key mixture at the 1/sqrt(hd) temperature, key/value permutation
invariance; SwiGLU on hand weights; a model whose layer outputs are zero maps
to softmax(W_lm . rmsnorm(E[x])); the cache-composition invariant (refresh
every step gives the no-cache trajectory).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from cached_masked_decoding_gb300 import synth
from cached_masked_decoding_gb300.configs import ModelConfig


@dataclasses.dataclass
class LayerWeights:
    attn_norm: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    ffn_norm: np.ndarray
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray


@dataclasses.dataclass
class Weights:
    cfg: ModelConfig
    embed: np.ndarray
    layers: list
    final_norm: np.ndarray
    lm_head: np.ndarray


def load_weights(cfg: ModelConfig, seed: int, random_norms: bool = False, layers=None) -> Weights:
    """Widen the seeded bf16 weights to float64.  ``layers`` limits which layers
    are materialised (others are None) for sampled checks of large models."""
    want = range(cfg.n_layers) if layers is None else layers
    lw = [None] * cfg.n_layers
    for l in want:
        t = {n: synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, n, l, random_norms)) for n in synth.LAYER_TENSORS}
        lw[l] = LayerWeights(**t)
    return Weights(
        cfg=cfg,
        embed=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "embed")),
        layers=lw,
        final_norm=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "final_norm", 0, random_norms)),
        lm_head=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "lm_head")),
    )


# --------------------------------------------------------------------------- pieces

def rms_norm(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm: h / sqrt(mean(h^2) + eps) * g, per row."""
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE. x: [n, H, hd]; dims j and j + hd/2 form a pair rotated by
    pos * theta^(-2j/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-(np.arange(half, dtype=np.float64) * 2.0) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, key_limit: np.ndarray | None = None) -> np.ndarray:
    """Non-causal multi-head attention, eq. 3. q: [n, H, hd]; k, v: [T, H, hd].
    key_limit (optional, [n]): query i sees keys t < key_limit[i] only."""
    hd = q.shape[-1]
    # per head: S = q k^T / sqrt(hd) as a batched matrix product [H][n][T]
    s = np.matmul(q.transpose(1, 0, 2), k.transpose(1, 2, 0)) / np.sqrt(hd)
    if key_limit is not None:
        hidden = np.arange(k.shape[0])[None, :] >= np.asarray(key_limit)[:, None]   # [n, T]
        s = np.where(hidden[None], -np.inf, s)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    # O = P V per head, back to [n][H][hd]
    return np.matmul(p, v.transpose(1, 0, 2)).transpose(1, 0, 2)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """W_d (silu(W_g x) * W_u x); weights are [out][in]."""
    return (silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def qkv(cfg: ModelConfig, lw: LayerWeights, h: np.ndarray, pos: np.ndarray):
    """Pre-norm projections of rows h at absolute positions pos; RoPE on q and k."""
    x = rms_norm(h, lw.attn_norm, cfg.norm_eps)
    n = h.shape[0]
    shp = (n, cfg.n_heads, cfg.head_dim)
    q = rope((x @ lw.wq.T).reshape(shp), pos, cfg.rope_theta)
    k = rope((x @ lw.wk.T).reshape(shp), pos, cfg.rope_theta)
    v = (x @ lw.wv.T).reshape(shp)
    return q, k, v


def block_key_limit(pos: np.ndarray, prompt_len: int, block: int) -> np.ndarray:
    """Block-causal visibility (BD3-LM style, the tutorial's section on caches;
    the dian8dian summary on block diffusion): a prompt position sees the
    prompt, a position of answer block j sees the prompt and blocks 0..j."""
    pos = np.asarray(pos)
    return np.where(pos < prompt_len, prompt_len, prompt_len + ((pos - prompt_len) // block + 1) * block)


def attn_ffn(cfg: ModelConfig, lw: LayerWeights, h: np.ndarray, q: np.ndarray,
             k_all: np.ndarray, v_all: np.ndarray, key_limit: np.ndarray | None = None) -> np.ndarray:
    """h += W_o Attn(q, K, V); h += SwiGLU(RMSNorm(h))."""
    o = attention(q, k_all, v_all, key_limit).reshape(h.shape[0], cfg.d_model)
    h = h + o @ lw.wo.T
    x = rms_norm(h, lw.ffn_norm, cfg.norm_eps)
    return h + swiglu(x, lw.wg, lw.wu, lw.wd)


@dataclasses.dataclass
class RowsForward:
    h_final: np.ndarray      # [n, d] residual stream after the last layer
    k: list                  # per layer: K context actually attended [T, H, hd]
    v: list
    h_layers: list           # per layer input (h_layers[0] = embedding), then the output


def forward_rows(w: Weights, tokens: np.ndarray, rows: np.ndarray,
                 k_ctx: list | None, v_ctx: list | None, keep_layers: bool = False,
                 skip_last_post_attn: bool = False, key_limit: np.ndarray | None = None) -> RowsForward:
    """Run the layer stack over the positions ``rows`` of one sequence.

    ``tokens`` is the whole canvas [T]; the K/V of the other positions come from
    ``k_ctx[l]`` / ``v_ctx[l]`` ([T, H, hd] per layer); the freshly computed K/V of
    ``rows`` replace theirs before attention.  With ``k_ctx=None`` every position
    must be in ``rows`` (a full-sequence forward).
    """
    cfg = w.cfg
    T = tokens.shape[0]
    rows = np.asarray(rows)
    h = w.embed[tokens[rows]]
    ks, vs, hl = [], [], [h.copy()] if keep_layers else []
    for l in range(cfg.n_layers):
        lw = w.layers[l]
        q, k, v = qkv(cfg, lw, h, rows)
        if k_ctx is None:
            if rows.shape[0] != T:
                raise ValueError("a forward without a cache must cover every position")
            k_all = np.empty((T, cfg.n_heads, cfg.head_dim))
            v_all = np.empty_like(k_all)
        else:
            k_all = k_ctx[l].copy()
            v_all = v_ctx[l].copy()
        k_all[rows] = k
        v_all[rows] = v
        ks.append(k_all)
        vs.append(v_all)
        if skip_last_post_attn and l == cfg.n_layers - 1:
            break
        h = attn_ffn(cfg, lw, h, q, k_all, v_all, key_limit)
        if keep_layers:
            hl.append(h.copy())
    return RowsForward(h_final=h, k=ks, v=vs, h_layers=hl)


@dataclasses.dataclass
class HeadStats:
    logits: np.ndarray    # [n, V]
    conf: np.ndarray      # [n] float64, largest softmax probability
    arg: np.ndarray       # [n] int, argmax (lowest id among equal maxima)
    margin: np.ndarray    # [n] top-1 minus top-2 logit


def lm_head(w: Weights, h_final: np.ndarray) -> HeadStats:
    """Final RMSNorm, LM head and per-row softmax maximum / argmax (Algorithm 2,
    steps 1-2).  conf = 1 / sum_v exp(l_v - l_max)."""
    x = rms_norm(h_final, w.final_norm, w.cfg.norm_eps)
    logits = x @ w.lm_head.T
    arg = np.argmax(logits, axis=-1)           # first index among maxima
    lmax = logits[np.arange(logits.shape[0]), arg]
    conf = 1.0 / np.exp(logits - lmax[:, None]).sum(axis=-1)
    part = np.partition(logits, -2, axis=-1)
    margin = part[:, -1] - part[:, -2]
    return HeadStats(logits=logits, conf=conf, arg=arg, margin=margin)
