"""Trajectory comparison of the GPU decoder against the CPU oracle.

Trajectory-sync rule (the stated tolerances of the method's parity bar): at
every step the oracle recomputes the step from the GPU's canvas.  Then

* the GPU's per-position max-prob must match the oracle's within ``TOL``
  (2e-3 absolute) at every MASK position of the block;
* the GPU's argmax must equal the oracle's, except where the oracle's
  top-1/top-2 logit margin is below ``TOL`` (an argmax near tie, counted);
* the GPU's commit must be exactly the selection rule applied to the GPU's own
  confidences and argmaxes (bit-exact selection given identical inputs);
* where the oracle's own confidences would select differently, the decision
  must sit within ``TOL`` of a decision boundary: a confidence within TOL of
  tau (or of the factor / budget boundary), or two ranked confidences within
  TOL of each other (a selection near tie, counted).

The oracle then adopts the GPU's commit and both continue.  Every run's counts
(decisions, near ties, argmax near ties) are kept in a ``Report``; with the
environment variable ``DLLM_PARITY_LOG`` set they are also appended to that
file as one JSON line per run.

Two drivers: ``run_synced`` walks Algorithm 1 from Python, one C call per
refresh and step; ``run_loop_synced`` lets the library's own loop
(``dllm_run``) walk it and follows it through the run hook, the oracle
running the same events (``oracle.sampler.Decoder.run``) in lockstep.
"""
import dataclasses
import json
import os

import numpy as np

from cached_masked_decoding_gb300 import binding
from oracle import sampler as OS

TOL = 2e-3


def conf_tol(cfg) -> float:
    """Max-prob tolerance: the stated 2e-3 for every model.  It holds because
    the split-precision path keeps q, K, V and the attention probabilities as
    hi/lo bf16 pairs."""
    return TOL


def to_gpu_rule(rule: OS.Rule):
    return binding.make_select(rule.policy, rule.tau, rule.k, rule.factor)


def decision_margin(rule: OS.Rule, conf: np.ndarray, elig: np.ndarray) -> float:
    """Distance (in confidence) of the rule's decision from its nearest boundary."""
    c = np.sort(conf[elig].astype(np.float64))[::-1]
    if c.size == 0:
        return np.inf
    gaps = np.diff(c) * -1 if c.size > 1 else np.array([np.inf])
    rank_gap = float(gaps.min()) if gaps.size else np.inf
    if rule.policy == OS.THRESHOLD:
        return min(float(np.abs(c - rule.tau).min()), rank_gap)
    if rule.policy in (OS.FIXED_K, OS.SCHEDULE):
        return rank_gap
    if rule.policy == OS.FACTOR:
        n = np.arange(1, c.size + 1)
        return min(float(np.abs((n + 1) * (1 - c) - rule.factor).min() / (c.size + 1)), rank_gap)
    e = 1 - c
    cs = np.cumsum(e)
    return min(float(np.abs(cs + e - 1).min() / (c.size + 1)), rank_gap)


class Report:
    def __init__(self):
        self.steps = 0
        self.refreshes = 0
        self.decisions = 0
        self.near_ties = 0
        self.arg_near_ties = 0
        self.max_conf_err = 0.0
        self.max_hidden_rel = 0.0

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k in ("steps", "refreshes", "decisions", "near_ties", "arg_near_ties",
                                               "max_conf_err", "max_hidden_rel")}

    def __repr__(self):
        return (f"steps={self.steps} refreshes={self.refreshes} decisions={self.decisions} "
                f"near_ties={self.near_ties} arg_near_ties={self.arg_near_ties} "
                f"max_conf_err={self.max_conf_err:.2e} max_hidden_rel={self.max_hidden_rel:.2e}")

    def check_bounds(self) -> None:
        """Near ties are rare by construction (a margin under 2e-3): a run
        that leans on many of them is not agreeing with the oracle."""
        assert self.near_ties <= max(2, self.steps // 10), f"too many selection near ties: {self}"
        assert self.arg_near_ties <= max(2, self.decisions // 100), f"too many argmax near ties: {self}"

    def log(self, **extra) -> None:
        path = os.environ.get("DLLM_PARITY_LOG")
        if not path:
            return
        rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], **self.as_dict(), **extra}
        with open(path, "a") as fh:
            fh.write(json.dumps(rec) + "\n")


def check_step(rep: Report, dec: OS.Decoder, rule: OS.Rule, j: int, x_before: np.ndarray, x_after: np.ndarray,
               conf_g: np.ndarray, arg_g: np.ndarray, h_g: np.ndarray | None, conf_o: np.ndarray,
               arg_o: np.ndarray, margin: np.ndarray, h_o: np.ndarray) -> None:
    """The trajectory-sync rule for one step of block j (see the module header)."""
    s = dec.block_start(j)
    elig = x_before[:, s:s + dec.B] == dec.cfg.mask_id
    rep.steps += 1
    if not elig.any():
        return
    err = np.abs(conf_g.astype(np.float64) - conf_o)[elig]
    rep.max_conf_err = max(rep.max_conf_err, float(err.max()))
    assert err.max() <= TOL, f"block {j} step {rep.steps}: max-prob error {err.max():.3e}"
    if h_g is not None:
        hg = h_g.astype(np.float64)
        rel = np.linalg.norm(hg - h_o, axis=-1) / np.linalg.norm(h_o, axis=-1)
        rep.max_hidden_rel = max(rep.max_hidden_rel, float(rel.max()))
        assert rel.max() <= 1e-2, f"final hidden relative error {rel.max():.3e}"
    mism = elig & (arg_g != arg_o)
    for i, k in zip(*np.nonzero(mism)):
        assert margin[i, k] < TOL, \
            f"argmax differs at block {j} seq {i} pos {k}: oracle top-1/top-2 margin {margin[i, k]:.3e} >= {TOL}"
    rep.arg_near_ties += int(mism.sum())
    for i in range(dec.b):
        sel_g = OS.select(rule, conf_g[i], elig[i])
        expect = x_before[i].copy()
        expect[s + np.flatnonzero(sel_g)] = arg_g[i, np.flatnonzero(sel_g)]
        np.testing.assert_array_equal(x_after[i], expect, err_msg="commit is not the rule on GPU conf")
        sel_o = OS.select(rule, conf_o[i].astype(np.float32), elig[i])
        rep.decisions += int(elig[i].sum())
        if not np.array_equal(sel_o, sel_g):
            dm = decision_margin(rule, conf_o[i], elig[i])
            assert dm < TOL, f"selection differs with decision margin {dm:.3e} >= {TOL} (seq {i}, block {j})"
            rep.near_ties += 1


def _step_rule(rule: OS.Rule, spb: int) -> OS.Rule:
    """The rule of a block's step spb: the scheduled rule counts k down."""
    if rule.policy == OS.SCHEDULE:
        return dataclasses.replace(rule, k=max(1, rule.k - spb))
    return rule


def run_synced(gpu: binding.State, dec: OS.Decoder, rule: OS.Rule, mode: str, check_hidden: bool = True,
               max_steps: int | None = None, max_blocks: int | None = None) -> Report:
    """Algorithm 1 driven from Python: one C call per refresh and step
    (optionally only the first max_blocks blocks, for long answers)."""
    rep = Report()
    n_blocks = dec.n_blocks if max_blocks is None else min(dec.n_blocks, max_blocks)
    cached = mode != "none"
    if cached:
        gpu.refresh()
        dec.refresh()
        rep.refreshes += 1
    for j in range(n_blocks):
        s = dec.block_start(j)
        spb = 0
        while True:
            x_before = gpu.tokens()
            np.testing.assert_array_equal(x_before, dec.x, err_msg="trajectories out of sync")
            if not (x_before[:, s:s + dec.B] == dec.cfg.mask_id).any():
                break
            step_rule = _step_rule(rule, spb)
            spb += 1
            gpu.step_ex(j, to_gpu_rule(step_rule), mode)
            x_after, conf_g, arg_g = gpu.read()
            conf_o, arg_o, margin, hb, _ = dec.compute(j)
            check_step(rep, dec, step_rule, j, x_before, x_after, conf_g, arg_g,
                       gpu.hidden() if check_hidden else None, conf_o, arg_o, margin, hb)
            dec.x = x_after.astype(np.int64).copy()
            if max_steps is not None and rep.steps >= max_steps:
                rep.log(mode=mode, driver="python", truncated=True)
                return rep
        if cached and j + 1 < n_blocks:
            gpu.refresh()
            dec.refresh()
            rep.refreshes += 1
    rep.check_bounds()
    rep.log(mode=mode, driver="python")
    return rep


def run_loop_synced(gpu: binding.State, dec: OS.Decoder, rule: OS.Rule, mode: str, refresh_interval: int = 0,
                    check_hidden: bool = True, ignore_refreshes: bool = False) -> tuple:
    """dllm_run (the library's own Algorithm 1 loop, the one the bench times)
    followed event by event through its run hook.  The oracle decoder runs
    the same loop (``Decoder.run``) in lockstep: every GPU event must be the
    oracle's next event (same kind, same block); each step is checked with the
    trajectory-sync rule and the oracle then continues from the GPU's canvas.
    With ``ignore_refreshes`` the GPU's refresh events are not matched (the
    oracle decoder is a no-cache one that the cached GPU run must reproduce).
    Returns (Report, dllm_run's stats)."""
    rep = Report()
    events = dec.run(rule, refresh_interval)
    box = {"started": False, "adopt": None, "x_before": gpu.tokens(), "exc": None, "spb": 0}

    def next_event():
        ev = events.send(box["adopt"]) if box["started"] else next(events)
        box["started"] = True
        box["adopt"] = None
        return ev

    def hook(event, j, spb):
        try:
            kind = "step" if event == binding.EVENT_STEP else "refresh"
            if kind == "refresh":
                rep.refreshes += 1
                if ignore_refreshes:
                    return 0
            ev = next_event()
            assert ev[0] == kind and ev[1] == j, \
                f"the GPU loop's event ({kind}, block {j}, step {spb}) is not the oracle's next {ev[:2]}"
            if kind == "step":
                out = ev[2]
                np.testing.assert_array_equal(box["x_before"], out.x_before, err_msg="trajectories out of sync")
                x_after, conf_g, arg_g = gpu.read()
                check_step(rep, dec, _step_rule(rule, spb), j, box["x_before"], x_after, conf_g, arg_g,
                           gpu.hidden() if check_hidden else None, out.conf, out.arg, out.margin, out.h_block)
                box["adopt"] = x_after.astype(np.int64)
                box["x_before"] = x_after
            return 0
        except BaseException as e:   # reported after dllm_run returns
            box["exc"] = e
            return 1

    gpu.set_run_hook(hook)
    try:
        stats = gpu.run(to_gpu_rule(rule), mode, refresh_interval=refresh_interval)
    except binding.DllmError:
        if box["exc"] is not None:
            raise box["exc"]
        raise
    finally:
        gpu.set_run_hook(None)
    if box["exc"] is not None:
        raise box["exc"]
    # the GPU loop ended: so must the oracle's
    try:
        ev = next_event()
    except StopIteration:
        ev = None
    assert ev is None, f"the GPU loop stopped before the oracle's event {ev[:2]}"
    assert stats["steps"] == rep.steps == dec.steps
    if not ignore_refreshes:
        assert stats["refreshes"] == rep.refreshes == dec.refreshes
    rep.check_bounds()
    rep.log(mode=mode, driver="dllm_run", refresh_interval=refresh_interval)
    return rep, stats
