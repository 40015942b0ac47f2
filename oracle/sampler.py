"""Oracle sampler: block-cached decoding loop and the position-selection rules.

TEST INFRASTRUCTURE ONLY (see package header).

Passages followed (zhongzhuzhou.org Fast-dLLM reading notes unless noted):

* ``Decoder.generate`` - Algorithm 1 (section 3, "block-wise cached decoding"):
  append L MASKs to the prompt; initialise K/V from the full context; walk the
  answer blocks left to right; while the current block holds MASK, recompute the
  current block and the suffix (PrefixCache) or only the current block
  (DualCache), let the queries read fresh and cached K/V, get candidates and
  confidences, pick positions with Algorithm 2 or 3 and fill them all at once;
  refresh the cached representations before moving to the next block.
  ``mode="none"`` recomputes every position every step (page 1, section on the
  KV cache: without a cache every step recomputes prompt and answer).
* ``select_threshold`` - Algorithm 2 (section 4): y_i = argmax, c_i = max prob,
  S = {c_i >= tau}; if S is empty take the single most confident position.
* ``select_factor`` - Algorithm 3 / eq. 13 (section 6): sort by confidence, keep
  the largest n with (n+1)(1 - c_(n)) < f, else the single best.
* ``select_budget`` - eq. 9 (section 5.1): the largest confidence-ordered prefix
  with sum_j eps_j + max_j eps_j < 1, else the single best.
* ``select_schedule`` - page 1's LLaDA low-confidence remasking inside a
  block: with k steps left, the (MASK count) // k most confident are kept.
* ``select_fixed_k`` - the fixed-count rule (page 1, opening paragraph: a fixed
  number of tokens per step; LLaDA's low-confidence remasking keeps the most
  confident predictions).
* ``staleness`` - Algorithm 4 of the notes (section 14), steps 4-5: fresh
  versus cached K/V rows (cosine per layer) and predictions (argmax
  agreement, max-prob difference) for the current block.
* ``llada_sample`` - page 1's LLaDA sampler (the tutorial's prose on one
  step from time t to s): a full bidirectional forward predicts every masked
  position, low-confidence remasking puts about s/t of them back under MASK
  (the least confident) and writes the rest, which never change afterwards.
* ``Decoder.run`` with ``refresh_interval`` - the refresh schedule separated
  from the block schedule (notes, section 11, Table 10's refresh intervals
  and the section's closing paragraph).

Readings where the pages are silent (each also listed in the design notes):
eligible positions are the MASK positions of the current block only; ties in
confidence go to the lowest position, ties in the argmax to the lowest token
id; fixed-k takes min(k, remaining); the refresh forward commits nothing; a
batch runs in lockstep (a finished sequence commits 0 in a step) and refreshes
together once every sequence has finished the block; decisions are taken in
float32 on the float32-rounded confidence.

Pins (tests/test_oracle_pins.py): the poker example (page 1 and page 2) and
the invariants - committed tokens never change, every step commits >= 1 while
MASK remains, tau > 1 reproduces ``llada_sample`` with one commit per step,
refreshing before every step reproduces the no-cache trajectory, a refresh
interval of at least B is the block-boundary schedule, at most B steps per
block, the tutorial's worked example of two steps keeping two tokens each.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import model as M

THRESHOLD, FIXED_K, FACTOR, BUDGET, SCHEDULE = 0, 1, 2, 3, 4


@dataclasses.dataclass(frozen=True)
class Rule:
    policy: int = THRESHOLD
    tau: float = 0.9
    k: int = 1
    factor: float = 1.0


def _order(conf32: np.ndarray, eligible: np.ndarray) -> np.ndarray:
    """Eligible positions sorted by descending confidence, ties by position."""
    idx = np.flatnonzero(eligible)
    return idx[np.lexsort((idx, -conf32[idx].astype(np.float64)))]


def select_threshold(conf32: np.ndarray, eligible: np.ndarray, tau: float) -> np.ndarray:
    sel = np.zeros(conf32.shape[0], dtype=bool)
    if not eligible.any():
        return sel
    t = np.float32(tau)
    sel = eligible & (conf32 >= t)
    if not sel.any():
        sel[_order(conf32, eligible)[0]] = True
    return sel


def select_fixed_k(conf32: np.ndarray, eligible: np.ndarray, k: int) -> np.ndarray:
    sel = np.zeros(conf32.shape[0], dtype=bool)
    sel[_order(conf32, eligible)[:max(0, k)]] = True
    return sel


def select_factor(conf32: np.ndarray, eligible: np.ndarray, factor: float) -> np.ndarray:
    sel = np.zeros(conf32.shape[0], dtype=bool)
    order = _order(conf32, eligible)
    if order.size == 0:
        return sel
    f = np.float32(factor)
    best = 0
    for n in range(1, order.size + 1):
        c_n = conf32[order[n - 1]]
        if np.float32(n + 1) * (np.float32(1.0) - c_n) < f:
            best = n
    sel[order[:max(best, 1)]] = True
    return sel


def select_budget(conf32: np.ndarray, eligible: np.ndarray) -> np.ndarray:
    sel = np.zeros(conf32.shape[0], dtype=bool)
    order = _order(conf32, eligible)
    if order.size == 0:
        return sel
    best = 0
    total = np.float32(0.0)
    for n in range(1, order.size + 1):
        e = np.float32(1.0) - conf32[order[n - 1]]   # the largest eps so far (sorted)
        total = np.float32(total + e)
        if np.float32(total + e) < np.float32(1.0):
            best = n
    sel[order[:max(best, 1)]] = True
    return sel


def select_schedule(conf32: np.ndarray, eligible: np.ndarray, steps_left: int) -> np.ndarray:
    """Page 1's LLaDA remasking schedule: with steps_left steps to go, keep the
    n_keep = (MASK count) // steps_left most confident predictions (possibly
    none this step)."""
    n_keep = int(eligible.sum()) // max(int(steps_left), 1)
    return select_fixed_k(conf32, eligible, n_keep)


def select(rule: Rule, conf32: np.ndarray, eligible: np.ndarray) -> np.ndarray:
    if rule.policy == THRESHOLD:
        return select_threshold(conf32, eligible, rule.tau)
    if rule.policy == FIXED_K:
        return select_fixed_k(conf32, eligible, rule.k)
    if rule.policy == FACTOR:
        return select_factor(conf32, eligible, rule.factor)
    if rule.policy == BUDGET:
        return select_budget(conf32, eligible)
    if rule.policy == SCHEDULE:            # rule.k: the steps left in the block
        return select_schedule(conf32, eligible, rule.k)
    raise ValueError(rule.policy)


@dataclasses.dataclass
class StepOut:
    block: int
    x_before: np.ndarray     # [b][T]
    conf: np.ndarray         # [b][B] float64
    conf32: np.ndarray       # [b][B] float32 (the deciding precision)
    arg: np.ndarray          # [b][B]
    margin: np.ndarray       # [b][B] top-1 minus top-2 logit
    h_block: np.ndarray      # [b][B][d] residual stream after the last layer
    selected: np.ndarray     # [b][B] bool
    committed: np.ndarray    # [b] count
    eligible: np.ndarray     # [b][B] bool, MASK positions of the block before the step


class Decoder:
    """Lockstep batch decoder following Algorithm 1 with one of three cache modes."""

    def __init__(self, w: M.Weights, prompts: np.ndarray, gen_len: int, block: int, mode: str,
                 mask: str = "full"):
        if mode not in ("none", "prefix", "dual"):
            raise ValueError(mode)
        if mask not in ("full", "block_causal"):
            raise ValueError(mask)
        self.mask = mask
        if gen_len % block != 0:
            raise ValueError("gen_len must be a multiple of block")
        self.w = w
        self.cfg = w.cfg
        self.b, self.P = prompts.shape
        self.gen = gen_len
        self.B = block
        self.T = self.P + gen_len
        self.mode = mode
        self.x = np.concatenate(
            [np.asarray(prompts, dtype=np.int64), np.full((self.b, gen_len), self.cfg.mask_id, dtype=np.int64)], axis=1)
        self.k_cache = [None] * self.b
        self.v_cache = [None] * self.b
        self.refreshes = 0
        self.steps = 0

    @property
    def n_blocks(self) -> int:
        return self.gen // self.B

    def block_start(self, j: int) -> int:
        return self.P + j * self.B

    def refresh(self) -> None:
        """Full-sequence forward that rewrites every cached K/V (Algorithm 1, steps 2 and 11)."""
        rows = np.arange(self.T)
        for i in range(self.b):
            fw = M.forward_rows(self.w, self.x[i], rows, None, None, skip_last_post_attn=True,
                                key_limit=self.key_limit(rows))
            self.k_cache[i] = fw.k
            self.v_cache[i] = fw.v
        self.refreshes += 1

    def key_limit(self, rows: np.ndarray):
        """Per-row key limits of the block-causal mask, or None (bidirectional)."""
        if self.mask == "full":
            return None
        return M.block_key_limit(rows, self.P, self.B)

    def rows_of(self, j: int) -> np.ndarray:
        s = self.block_start(j)
        if self.mode == "dual":
            return np.arange(s, s + self.B)
        if self.mode == "prefix":
            return np.arange(s, self.T)
        return np.arange(self.T)

    def compute(self, j: int, keep_layers: bool = False):
        """Forward of the rows this mode recomputes; LM head on the block rows."""
        s = self.block_start(j)
        rows = self.rows_of(j)
        conf = np.zeros((self.b, self.B))
        arg = np.zeros((self.b, self.B), dtype=np.int64)
        margin = np.zeros((self.b, self.B))
        hb = np.zeros((self.b, self.B, self.cfg.d_model))
        layers = []
        for i in range(self.b):
            if self.mode == "none":
                fw = M.forward_rows(self.w, self.x[i], rows, None, None, keep_layers=keep_layers,
                                    key_limit=self.key_limit(rows))
            else:
                fw = M.forward_rows(self.w, self.x[i], rows, self.k_cache[i], self.v_cache[i],
                                    keep_layers=keep_layers, key_limit=self.key_limit(rows))
            sel = (rows >= s) & (rows < s + self.B)
            hs = fw.h_final[sel]
            st = M.lm_head(self.w, hs)
            conf[i], arg[i], margin[i], hb[i] = st.conf, st.arg, st.margin, hs
            layers.append(fw.h_layers)
        return conf, arg, margin, hb, layers

    def eligible(self, j: int) -> np.ndarray:
        s = self.block_start(j)
        return self.x[:, s:s + self.B] == self.cfg.mask_id

    def step(self, j: int, rule: Rule) -> StepOut:
        x_before = self.x.copy()
        conf, arg, margin, hb, _ = self.compute(j)
        conf32 = conf.astype(np.float32)
        elig = self.eligible(j)
        sel = np.zeros_like(elig)
        s = self.block_start(j)
        for i in range(self.b):
            sel[i] = select(rule, conf32[i], elig[i])
            pos = np.flatnonzero(sel[i])
            self.x[i, s + pos] = arg[i, pos]
        self.steps += 1
        return StepOut(j, x_before, conf, conf32, arg, margin, hb, sel, sel.sum(axis=1), elig)

    def run(self, rule: Rule, refresh_interval: int = 0, max_steps: int | None = None):
        """Algorithm 1 as a stream of events, in the order the loop takes them.

        Yields ``("refresh", j)`` after each cache refresh (j = the block the
        loop is in, 0 for the prefill) and ``("step", j, StepOut)`` after each
        denoise step.  A consumer may ``send`` a canvas [b][T] back in reply to
        a step event; the decoder then continues from that canvas instead of
        its own commit (used to follow another decoder's trajectory).

        ``refresh_interval`` r separates the refresh schedule from the block
        schedule (zhongzhuzhou.org notes, section 11, Table 10 and the closing
        paragraph of the section): with r > 0 the cached K/V are also
        refreshed before every r-th step inside a block (before steps r, 2r,
        ... counted from the block's first step, which follows the
        block-boundary refresh); r = 0 refreshes at block boundaries only.
        """
        cached = self.mode != "none"
        if cached:
            self.refresh()
            yield ("refresh", 0)
        n = 0
        for j in range(self.n_blocks):
            spb = 0
            while self.eligible(j).any():
                if cached and refresh_interval > 0 and spb > 0 and spb % refresh_interval == 0:
                    self.refresh()
                    yield ("refresh", j)
                # the scheduled rule counts its k down within each block
                r = dataclasses.replace(rule, k=max(1, rule.k - spb)) if rule.policy == SCHEDULE else rule
                out = self.step(j, r)
                adopt = yield ("step", j, out)
                if adopt is not None:
                    self.x = np.asarray(adopt, dtype=np.int64).copy()
                spb += 1
                n += 1
                if max_steps is not None and n >= max_steps:
                    return
            if cached and j < self.n_blocks - 1:
                self.refresh()
                yield ("refresh", j)

    def generate(self, rule: Rule, refresh_interval: int = 0, max_steps: int | None = None):
        """Algorithm 1 (section 3).  Returns (answer tokens [b][gen], list of StepOut)."""
        trace = [ev[2] for ev in self.run(rule, refresh_interval, max_steps) if ev[0] == "step"]
        return self.x[:, self.P:].copy(), trace


def staleness(dec: Decoder, j: int) -> dict:
    """Fresh versus cached representations and predictions for block j of the
    current canvas (zhongzhuzhou.org notes, section 14, Algorithm 4 steps 4-5;
    section 3 on what DualCache freezes between refreshes).

    fresh: the K/V a full forward over the current canvas would cache.
    k_cos[l], v_cos[l]: mean over sequences, heads and the positions outside
    the block of cos(cached row, fresh row).  agree: fraction of the block's
    MASK positions whose argmax from the cache equals the argmax without a
    cache; max_dconf: the largest max-prob difference there.
    """
    cfg = dec.cfg
    s = dec.block_start(j)
    L, T = cfg.n_layers, dec.T
    outside = np.ones(T, dtype=bool)
    outside[s:s + dec.B] = False
    sums = np.zeros((2, L))
    count = 0
    for i in range(dec.b):
        fw = M.forward_rows(dec.w, dec.x[i], np.arange(T), None, None, skip_last_post_attn=True)
        for kind, (cached, fresh) in enumerate(((dec.k_cache[i], fw.k), (dec.v_cache[i], fw.v))):
            for l in range(L):
                c, f = cached[l][outside], fresh[l][outside]          # [positions, H, hd]
                cos = (c * f).sum(-1) / np.sqrt((c * c).sum(-1) * (f * f).sum(-1))
                sums[kind, l] += cos.sum()
        count += int(outside.sum()) * cfg.n_heads
    conf_c, arg_c, _, _, _ = dec.compute(j)
    none = Decoder(dec.w, dec.x[:, :dec.P], dec.gen, dec.B, "none")
    none.x = dec.x.copy()
    conf_f, arg_f, _, _, _ = none.compute(j)
    elig = dec.eligible(j)
    agree = float((arg_c == arg_f)[elig].mean()) if elig.any() else 1.0
    dconf = float(np.abs(conf_c - conf_f)[elig].max()) if elig.any() else 0.0
    return {"k_cos": sums[0] / count, "v_cos": sums[1] / count, "agree": agree, "max_dconf": dconf}


def tau_bar(trace, b: int) -> np.ndarray:
    """Average tokens committed per step, per sequence, over the steps in which
    the sequence still had MASK in the current block."""
    committed = np.zeros(b)
    active = np.zeros(b)
    for st in trace:
        active += st.eligible.any(axis=1)
        committed += st.committed
    return committed / np.maximum(active, 1)


def llada_remask_count(masked: int, steps: int, k: int) -> int:
    """How many of this step's predictions go back under MASK in page 1's
    LLaDA sampler.  The step runs from time t = (steps - k) / steps to
    s = (steps - k - 1) / steps and re-masks about s/t of the positions that
    were masked: ceil(masked * s / t) of them, in exact integer arithmetic
    (so that the positions kept, masked minus this, spread the remaining MASKs
    evenly over the remaining steps, rounded down)."""
    left = steps - k
    return -((-masked * (left - 1)) // left)


def llada_sample(w: M.Weights, prompt: np.ndarray, gen_len: int, steps: int) -> np.ndarray:
    """Page 1's LLaDA sampler (tutorial, section on what one step does): each
    step one full bidirectional forward predicts every masked position, and
    low-confidence remasking puts the least confident predictions back under
    MASK (``llada_remask_count`` of them) while the rest are written; a written
    token is never changed again.  Ties: among equal confidences the later
    position is re-masked first (so the earlier one is kept)."""
    cfg = w.cfg
    P = int(np.asarray(prompt).shape[0])
    x = np.concatenate([np.asarray(prompt, dtype=np.int64), np.full(gen_len, cfg.mask_id, dtype=np.int64)])
    for k in range(steps):
        masked = np.flatnonzero(x == cfg.mask_id)
        if masked.size == 0:
            break
        pred = M.lm_head(w, M.forward_rows(w, x, np.arange(x.shape[0]), None, None).h_final)
        c32 = pred.conf.astype(np.float32)
        back = llada_remask_count(masked.size, steps, k)
        # least confident first; among equals the higher position first
        worst_first = masked[np.lexsort((-masked, c32[masked].astype(np.float64)))]
        write = worst_first[back:]
        x[write] = pred.arg[write]
    return x[P:]
