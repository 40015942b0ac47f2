"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (fixtures under tests/golden/ with their citations), closed forms,
brute force over tiny joint distributions, and invariants of the sampler.
"""
import itertools
import json
import os

import numpy as np
import pytest

from cached_masked_decoding_gb300 import configs, roofline, synth
from oracle import model as M
from oracle import sampler as S
from oracle import theory as TH

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# --------------------------------------------------------------------------- theory

def test_worked_example_product_tv_and_greedy():
    g = golden("worked_example.json")
    p = np.array(g["joint"])
    ms = TH.marginals(p)
    assert ms[0][0] == pytest.approx(g["marginal_top"]) and ms[1][0] == pytest.approx(g["marginal_top"])
    q = TH.product_of_marginals(p)
    np.testing.assert_allclose(q, np.array(g["product"]), atol=1e-12)
    assert TH.tv(p, q) == pytest.approx(g["tv"], abs=1e-12)
    assert list(TH.marginal_argmax(p)) == g["greedy"]
    assert sorted(TH.argmax_strings(p)) == sorted(tuple(x) for x in g["joint_argmax"])
    # reverse KL is infinite: q gives mass to (1,1) where p has none (section 5.2)
    assert TH.kl(q, p) == float("inf")


def _concentrated_joint(rng, n, V, delta, alpha):
    xs = tuple(rng.integers(0, V, size=n))
    p = rng.dirichlet(np.full(V ** n, alpha)).reshape((V,) * n) * delta
    p[xs] += 1.0 - delta
    return p


def _joint_samples(seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for n in (1, 2, 3):
        for V in (2, 3, 4):
            for alpha in (0.05, 0.3, 1.0):
                for _ in range(60):
                    out.append(rng.dirichlet(np.full(V ** n, alpha)).reshape((V,) * n))
                for delta in (0.02, 0.1, 0.2, 0.3, 0.45):
                    for _ in range(25):
                        out.append(_concentrated_joint(rng, n, V, delta, alpha))
    return out


SAMPLES = _joint_samples()


def test_theorem1_brute_force():
    applied = 0
    for p in SAMPLES:
        if not TH.theorem1_applies(p):
            continue
        applied += 1
        xs = TH.marginal_argmax(p)
        assert TH.argmax_strings(p) == [xs]                      # eq. 8, joint side (unique)
        assert TH.argmax_strings(TH.product_of_marginals(p)) == [xs]   # eq. 8, product side
    assert applied > 300


def test_theorem1_proof_steps_union_bound_and_single_position():
    for p in SAMPLES:
        e = TH.eps_per_position(p)
        xs = TH.marginal_argmax(p)
        if e.max() >= 0.5:
            continue
        assert p[xs] >= 1.0 - e.sum() - 1e-12                     # eq. 6 (union bound)
        others = p.copy()
        others[xs] = -1
        assert others.max() <= e.max() + 1e-12                    # eq. 7


def test_theorem1_is_tight():
    # the family needs n >= 2: each single-one string then holds less than half the mass
    for n in (2, 3, 4):
        for eta in (1e-3, 1e-2):
            p = TH.tightness_family(n, eta)
            assert p.sum() == pytest.approx(1.0)
            e = TH.eps_per_position(p)
            assert np.all(e < 0.5)                                 # every marginal still prefers 0
            assert TH.marginal_argmax(p) == (0,) * n
            assert (n + 1) * e.max() > 1.0                         # just beyond the bound
            assert (0,) * n not in TH.argmax_strings(p)            # and the joint argmax moves


def test_eq9_nonuniform_budget_is_sufficient():
    hits = 0
    for p in SAMPLES:
        if TH.eq9_holds(p):
            hits += 1
            assert TH.argmax_strings(p) == [TH.marginal_argmax(p)]
    assert hits > 300
    # eq. 9 is looser than the uniform condition: some samples satisfy 9 but not (n+1)eps<=1
    assert any(TH.eq9_holds(p) and not TH.theorem1_applies(p) for p in SAMPLES)


def test_tv_bound_eq10():
    for p in SAMPLES:
        e = TH.eps_per_position(p).max()
        q = TH.product_of_marginals(p)
        assert TH.tv(p, q) <= TH.tv_bound(p.ndim, e) + 1e-12


def test_kl_is_total_correlation_and_chain_rule_eq11():
    for p in SAMPLES[::7]:
        q = TH.product_of_marginals(p)
        d = TH.kl(p, q)
        assert d == pytest.approx(TH.total_correlation(p), abs=1e-10)
        assert d == pytest.approx(TH.chain_mutual_information(p), abs=1e-10)


def test_kl_bound_eq12():
    for p in SAMPLES:
        e = TH.eps_per_position(p).max()
        V = p.shape[0]
        if e > 0.5 or V < 2:
            continue
        assert TH.kl(p, TH.product_of_marginals(p)) <= TH.kl_bound(p.ndim, e, V) + 1e-12


def test_theorem_arithmetic_printed_on_the_pages():
    g = golden("theorem_arithmetic.json")
    a = g["three_at_095"]
    assert (a["n"] + 1) * a["eps"] == pytest.approx(a["lhs"]) and ((a["n"] + 1) * a["eps"] <= 1) == a["holds"]
    n_max = max(n for n in range(1, 100) if (n + 1) * 0.1 <= 1 + 1e-12)
    assert n_max == g["eps_01_max_n"]


# --------------------------------------------------------------------------- selection

def test_poker_example_one_step_vs_threshold_rule():
    g = golden("poker.json")
    p = np.array(g["joint"])
    ms = TH.marginals(p)
    np.testing.assert_allclose(np.array(ms), np.array(g["marginals"]))
    q = TH.product_of_marginals(p)
    valid = p > 0
    assert q[valid].sum() == pytest.approx(g["one_step_valid_probability"])
    assert (p.ndim + 1) * g["theorem_eps"] == pytest.approx(g["theorem_lhs"])
    # Algorithm 2 at tau = 0.9 on the table model: marginals given the committed tokens.
    rule = S.Rule(S.THRESHOLD, 0.9)
    x = [-1, -1]
    steps = 0
    while -1 in x:
        cond = p.copy()
        for j, t in enumerate(x):
            if t >= 0:
                idx = [slice(None)] * 2
                keep = np.zeros(2, dtype=bool)
                keep[t] = True
                idx[j] = ~keep
                cond[tuple(idx)] = 0
        cond /= cond.sum()
        cm = TH.marginals(cond)
        conf = np.array([m.max() for m in cm], dtype=np.float32)
        arg = [int(np.argmax(m)) for m in cm]
        elig = np.array([t < 0 for t in x])
        sel = S.select(rule, conf, elig)
        if steps == 0:
            assert sel.sum() == 1                                  # commits one, not both
        for j in np.flatnonzero(sel):
            x[j] = arg[j]
        steps += 1
    assert steps == 2
    assert p[tuple(x)] > 0                                        # a valid hand: validity 1.0
    assert g["two_step_valid_probability"] == 1.0


def test_threshold_rule_cases():
    c = np.array([0.95, 0.5, 0.91, 0.2], dtype=np.float32)
    e = np.array([True, True, True, True])
    assert S.select_threshold(c, e, 0.9).tolist() == [True, False, True, False]
    # comparison is >= (Algorithm 2, step 3)
    c2 = np.array([0.9, 0.1], dtype=np.float32)
    assert S.select_threshold(c2, np.array([True, True]), float(np.float32(0.9))).tolist() == [True, False]
    # fallback: single most confident, ties to the lowest position
    c3 = np.array([0.4, 0.6, 0.6, 0.1], dtype=np.float32)
    assert S.select_threshold(c3, e, 0.9).tolist() == [False, True, False, False]
    # committed positions are not eligible even when confident
    e2 = np.array([False, True, True, True])
    assert S.select_threshold(c, e2, 0.9).tolist() == [False, False, True, False]
    # nothing eligible: nothing selected, no fallback
    assert not S.select_threshold(c, np.zeros(4, dtype=bool), 0.9).any()
    # tau > 1 never meets the threshold: always exactly one
    assert S.select_threshold(np.ones(4, dtype=np.float32), e, 1.5).sum() == 1


def test_fixed_k_and_factor_and_budget_cases():
    c = np.array([0.5, 0.99, 0.7, 0.99, 0.2], dtype=np.float32)
    e = np.ones(5, dtype=bool)
    assert np.flatnonzero(S.select_fixed_k(c, e, 2)).tolist() == [1, 3]
    assert np.flatnonzero(S.select_fixed_k(c, e, 10)).tolist() == [0, 1, 2, 3, 4]
    # factor f=1: n=1: 2*0.01<1 ok; n=2: 3*0.01<1 ok; n=3 (0.7): 4*0.3=1.2 no; n=4 (0.5): 5*0.5 no
    assert np.flatnonzero(S.select_factor(c, e, 1.0)).tolist() == [1, 3]
    # f=3: n=3: 1.2<3 ok; n=4: 2.5<3 ok; n=5 (0.2): 6*0.8=4.8 no -> largest n = 4
    assert np.flatnonzero(S.select_factor(c, e, 3.0)).tolist() == [0, 1, 2, 3]
    # f tiny: fallback to the single best (lowest position among the ties)
    assert np.flatnonzero(S.select_factor(c, e, 1e-6)).tolist() == [1]
    # eq. 9 budget: eps sorted 0.01, 0.01, 0.3, 0.5, 0.8; n=2: 0.02+0.01<1; n=3: 0.32+0.3<1; n=4: 0.82+0.5>=1
    assert np.flatnonzero(S.select_budget(c, e)).tolist() == [1, 2, 3]


def test_factor_rule_at_f1_matches_theorem_condition():
    # For f = 1 the factor rule's test (n+1)(1-c_(n)) < 1 is the theorem's (n+1)eps <= 1
    # with eps slightly above 1 - c_(n) (section 6).
    rng = np.random.default_rng(3)
    for _ in range(200):
        c = rng.uniform(0.5, 1.0, size=12).astype(np.float32)
        e = np.ones(12, dtype=bool)
        n = int(S.select_factor(c, e, 1.0).sum())
        cs = np.sort(c)[::-1]
        ok = [(m + 1) * (1 - float(cs[m - 1])) < 1 for m in range(1, 13)]
        expect = max([m for m in range(1, 13) if ok[m - 1]], default=1)
        assert n == expect


# --------------------------------------------------------------------------- model pieces

def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(0)
    h = rng.standard_normal((3, 64))
    g = np.ones(64)
    y = M.rms_norm(h, g, 0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(M.rms_norm(5.0 * h, g, 0.0), y, rtol=1e-12)
    eps = 0.3
    ye = M.rms_norm(h, g, eps)
    ms = (h * h).mean(-1)
    np.testing.assert_allclose((ye * ye).mean(-1), ms / (ms + eps), rtol=1e-12)
    g2 = rng.standard_normal(64)
    np.testing.assert_allclose(M.rms_norm(h, g2, 0.0), y * g2, rtol=1e-12)


def test_rope_closed_forms():
    theta = 1e4
    x = np.zeros((1, 1, 4))
    x[0, 0, 0] = 1.0
    p = 3
    y = M.rope(x, np.array([p]), theta)[0, 0]
    # pairs are (0, 2) and (1, 3); pair 0 turns by p * theta^0 = p radians
    np.testing.assert_allclose(y, [np.cos(p), 0.0, np.sin(p), 0.0], atol=1e-15)
    x = np.zeros((1, 1, 4))
    x[0, 0, 1] = 1.0
    y = M.rope(x, np.array([p]), theta)[0, 0]
    w = p * theta ** (-2.0 / 4)
    np.testing.assert_allclose(y, [0.0, np.cos(w), 0.0, np.sin(w)], atol=1e-15)
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 2, 8))
    np.testing.assert_allclose(M.rope(v, np.zeros(5), theta), v)
    r = M.rope(v, np.arange(5) * 7.0, theta)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(v, axis=-1), rtol=1e-12)
    # relative-position property: <R(m) q, R(n) k> depends on m - n only
    q = rng.standard_normal((1, 1, 8))
    k = rng.standard_normal((1, 1, 8))
    a = (M.rope(q, np.array([11.0]), theta) * M.rope(k, np.array([4.0]), theta)).sum()
    b = (M.rope(q, np.array([7.0]), theta) * M.rope(k, np.array([0.0]), theta)).sum()
    assert a == pytest.approx(b, rel=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    T, H, hd = 9, 2, 16
    v = rng.standard_normal((T, H, hd))
    k_same = np.repeat(rng.standard_normal((1, H, hd)), T, axis=0)
    q = rng.standard_normal((3, H, hd))
    np.testing.assert_allclose(M.attention(q, k_same, v), np.broadcast_to(v.mean(0), (3, H, hd)), rtol=1e-12)
    # two keys: weights exp(s_i / sqrt(hd)) / sum
    k2 = np.zeros((2, 1, 4))
    k2[0, 0, 0] = 2.0
    v2 = np.array([[[1.0, 0, 0, 0]], [[0, 1.0, 0, 0]]])
    q2 = np.array([[[1.0, 0, 0, 0]]])
    w0 = np.exp(2.0 / 2.0) / (np.exp(2.0 / 2.0) + 1.0)
    np.testing.assert_allclose(M.attention(q2, k2, v2)[0, 0], [w0, 1 - w0, 0, 0], rtol=1e-12)
    # non-causal: a joint permutation of keys and values changes nothing
    k = rng.standard_normal((T, H, hd))
    perm = rng.permutation(T)
    np.testing.assert_allclose(M.attention(q, k[perm], v[perm]), M.attention(q, k, v), rtol=1e-12)


# silu(t) = t * sigmoid(t) at fixed points: sigmoid(1) = e / (1 + e) and
# sigmoid(-2) = 1 / (1 + e^2), as published decimal constants.
SILU_1 = 0.7310585786300049
SILU_M2 = -0.2384058440442351


def test_silu_fixed_values():
    np.testing.assert_allclose(M.silu(np.array([1.0, -2.0, 0.0])), [SILU_1, SILU_M2, 0.0], rtol=1e-15, atol=0)
    # silu(t) - silu(-t) = t  (sigmoid(t) + sigmoid(-t) = 1)
    t = np.linspace(-6, 6, 13)
    np.testing.assert_allclose(M.silu(t) - M.silu(-t), t, atol=1e-14)


def test_swiglu_hand_weights():
    x = np.array([[1.0, -2.0]])
    wg = np.array([[1.0, 0.0], [0.0, 1.0]])
    wu = np.array([[2.0, 0.0], [0.0, 1.0]])
    wd = np.array([[1.0, 1.0]])
    # W_d (silu(W_g x) * W_u x) = silu(1) * 2 + silu(-2) * (-2)
    expect = SILU_1 * 2.0 + SILU_M2 * (-2.0)
    assert M.swiglu(x, wg, wu, wd)[0, 0] == pytest.approx(expect, rel=1e-14)


def _hand_cfg(**kw):
    base = dict(name="hand", n_layers=1, d_model=4, n_heads=2, head_dim=2, d_ffn=4, vocab=5, norm_eps=0.0)
    base.update(kw)
    return configs.ModelConfig(**base)


COS1, SIN1 = 0.5403023058681398, 0.8414709848078965       # cos(1 rad), sin(1 rad)


def test_qkv_hand_model():
    """A one-layer, d = 4, two-head (hd = 2) model whose q, k and v come out of
    distinct weights (W_q = I, W_k = 2I, W_v = 3I): RMSNorm scales a unit
    basis row e_c to 2 e_c; RoPE turns q and k of a head by pos * theta^0 =
    pos radians at absolute position pos, and leaves v alone; column c feeds
    head c // 2."""
    cfg = _hand_cfg()
    eye = np.eye(4)
    z = np.zeros((4, 4))
    lw = M.LayerWeights(attn_norm=np.ones(4), wq=eye, wk=2 * eye, wv=3 * eye, wo=z, ffn_norm=np.ones(4),
                        wg=z, wu=z, wd=z)
    h = np.array([[1.0, 0.0, 0.0, 0.0], [0.0, 0.0, 1.0, 0.0], [1.0, 0.0, 0.0, 0.0]])
    pos = np.array([1, 1, 0])
    q, k, v = M.qkv(cfg, lw, h, pos)
    assert q.shape == k.shape == v.shape == (3, 2, 2)
    # row 0: head 0 holds (2, 0), turned by 1 rad; head 1 is zero
    np.testing.assert_allclose(q[0], [[2 * COS1, 2 * SIN1], [0, 0]], atol=1e-15)
    np.testing.assert_allclose(k[0], [[4 * COS1, 4 * SIN1], [0, 0]], atol=1e-15)
    np.testing.assert_allclose(v[0], [[6.0, 0.0], [0, 0]], atol=1e-15)        # no rotation of v
    # row 1: the same vector in head 1
    np.testing.assert_allclose(q[1], [[0, 0], [2 * COS1, 2 * SIN1]], atol=1e-15)
    np.testing.assert_allclose(k[1], [[0, 0], [4 * COS1, 4 * SIN1]], atol=1e-15)
    np.testing.assert_allclose(v[1], [[0, 0], [6.0, 0.0]], atol=1e-15)
    # row 2: position 0 turns nothing
    np.testing.assert_allclose(q[2], [[2.0, 0.0], [0, 0]], atol=1e-15)
    np.testing.assert_allclose(k[2], [[4.0, 0.0], [0, 0]], atol=1e-15)


def test_lm_head_hand_logits_margin_and_ties():
    """Final RMSNorm of an all-ones row is the row itself (eps 0), so each
    logit is the sum of its LM-head row: logits (1, 4, 3.5, 3.25, -2) give the
    argmax 1 and a top-1/top-2 margin of 0.5; an equal top pair gives margin 0
    and the lower id."""
    cfg = _hand_cfg()
    rows = np.array([1.0, 4.0, 3.5, 3.25, -2.0])
    lm = np.zeros((5, 4))
    lm[:, 0] = rows
    w = M.Weights(cfg=cfg, embed=np.zeros((6, 4)), layers=[], final_norm=np.ones(4), lm_head=lm)
    st = M.lm_head(w, np.ones((1, 4)))
    np.testing.assert_allclose(st.logits[0], rows, atol=0)
    assert st.arg[0] == 1 and st.margin[0] == 0.5
    lm[3, 0] = 4.0
    st = M.lm_head(w, np.ones((1, 4)))
    assert st.arg[0] == 1 and st.margin[0] == 0.0
    # a dominant logit: confidence 1 / (1 + 4 e^-40) to double precision
    lm[:, 0] = [0.0, 40.0, 0.0, 0.0, 0.0]
    st = M.lm_head(w, np.ones((1, 4)))
    assert st.conf[0] == pytest.approx(1.0, abs=1e-16) and st.margin[0] == 40.0


def _tiny_weights(random_norms=False, cfg=configs.TINY_SPREAD):
    return M.load_weights(cfg, 0, random_norms=random_norms)


def test_zero_layers_reduce_to_embedding_head():
    w = _tiny_weights(random_norms=True)
    for lw in w.layers:
        lw.wo[:] = 0.0
        lw.wd[:] = 0.0
    tok = synth.prompts(w.cfg, 0, 1, 12)[0]
    fw = M.forward_rows(w, tok, np.arange(12), None, None)
    np.testing.assert_allclose(fw.h_final, w.embed[tok])
    st = M.lm_head(w, fw.h_final)
    x = w.embed[tok]
    x = x / np.sqrt((x * x).mean(-1, keepdims=True) + w.cfg.norm_eps) * w.final_norm
    logits = x @ w.lm_head.T
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    np.testing.assert_allclose(st.conf, p.max(-1), rtol=1e-12)
    np.testing.assert_array_equal(st.arg, p.argmax(-1))


def test_lm_head_one_hot_dominant_and_ties():
    cfg = configs.TINY
    w = _tiny_weights(cfg=cfg)
    w.lm_head[:] = 0.0
    w.lm_head[7, :] = 50.0
    h = np.ones((1, cfg.d_model))
    st = M.lm_head(w, h)
    assert st.arg[0] == 7 and st.conf[0] == pytest.approx(1.0)
    w.lm_head[:] = 0.0
    st = M.lm_head(w, h)
    assert st.arg[0] == 0 and st.conf[0] == pytest.approx(1.0 / cfg.vocab)


# --------------------------------------------------------------------------- sampler invariants

@pytest.fixture(scope="module")
def tiny_w():
    return _tiny_weights(random_norms=True)


def _run(w, mode, rule, P=16, gen=32, block=8, b=1, **kw):
    pr = synth.prompts(w.cfg, 0, b, P)
    dec = S.Decoder(w, pr, gen, block, mode)
    toks, trace = dec.generate(rule, **kw)
    return dec, toks, trace


@pytest.mark.parametrize("mode", ["none", "prefix", "dual"])
def test_invariants_never_rewrite_progress_and_step_bound(tiny_w, mode):
    dec, toks, trace = _run(tiny_w, mode, S.Rule(S.THRESHOLD, 0.9))
    assert (toks != tiny_w.cfg.mask_id).all()
    steps_per_block = np.zeros(dec.n_blocks, dtype=int)
    for st in trace:
        steps_per_block[st.block] += 1
        assert st.committed.sum() >= 1
        after = st.x_before.copy()
        s = dec.block_start(st.block)
        for i in range(dec.b):
            pos = np.flatnonzero(st.selected[i])
            assert (st.x_before[i, s + pos] == tiny_w.cfg.mask_id).all()   # only MASK is written
            after[i, s + pos] = st.arg[i, pos]
        committed_before = st.x_before != tiny_w.cfg.mask_id
        assert (after[committed_before] == st.x_before[committed_before]).all()
    assert (steps_per_block <= dec.B).all()
    # the prompt is never touched
    assert (dec.x[:, :dec.P] == synth.prompts(tiny_w.cfg, 0, 1, 16)).all()


def test_tau_above_one_is_llada_one_per_step(tiny_w):
    P, gen = 12, 16
    pr = synth.prompts(tiny_w.cfg, 0, 1, P)
    dec = S.Decoder(tiny_w, pr, gen, gen, "none")
    toks, trace = dec.generate(S.Rule(S.THRESHOLD, 1.5))
    assert len(trace) == gen and all(st.committed.sum() == 1 for st in trace)
    ref = S.llada_sample(tiny_w, pr[0], gen, gen)
    np.testing.assert_array_equal(toks[0], ref)


@pytest.mark.parametrize("steps", [4, 7, 16, 20])
def test_schedule_rule_is_llada_sampler(tiny_w, steps):
    """Page 1's LLaDA sampler (whole answer, full forward, n_keep = remaining
    MASKs spread over the remaining steps) written out on its own, against the
    block decoder with the scheduled rule, one block covering the answer and
    no cache: the same tokens, exactly `steps` steps (more steps than MASKs
    leave the early steps empty)."""
    P, gen = 12, 16
    pr = synth.prompts(tiny_w.cfg, 3, 1, P)
    dec = S.Decoder(tiny_w, pr, gen, gen, "none")
    toks, trace = dec.generate(S.Rule(S.SCHEDULE, k=steps))
    assert len(trace) == steps
    assert sum(int(st.committed.sum()) for st in trace) == gen
    np.testing.assert_array_equal(toks[0], S.llada_sample(tiny_w, pr[0], gen, steps))


def test_llada_remask_count_worked_example():
    """The tutorial's worked example ('the tea is cold'): four positions, two
    steps, two tokens kept per step; tea's 0.3 at step 1 puts it back under
    MASK, and at step 2 everything left is written."""
    g = golden("tea_is_cold.json")
    m = g["gen_len"]
    kept = []
    for k in range(g["steps"]):
        back = S.llada_remask_count(m, g["steps"], k)
        kept.append(m - back)
        m = back
    assert kept == g["kept_per_step"] and m == 0
    # the selection at step 1: tea (0.3) is among the re-masked, the and is are kept
    words = ["the", "tea", "is", "cold"]
    conf = np.array([0.9, g["tea_confidence"]["step_1"], 0.8, 0.2], dtype=np.float32)
    sel = S.select_schedule(conf, np.ones(4, dtype=bool), g["steps"])
    assert [w for w, s_ in zip(words, sel) if s_] == g["kept_at_step_1"]


def test_llada_remask_count_spreads_evenly():
    """Keeping masked - remask positions spreads the remaining MASKs evenly
    over the remaining steps, rounded down, and the last step writes them all."""
    for steps in range(1, 25):
        for m in range(0, 70):
            for k in range(steps):
                kept = m - S.llada_remask_count(m, steps, k)
                assert kept * (steps - k) <= m < (kept + 1) * (steps - k)
            assert S.llada_remask_count(m, steps, steps - 1) == 0


def test_attention_key_limit_closed_forms():
    """A key limit of T is the unmasked attention; a limit of 1 returns v[0]."""
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((5, 2, 8)), rng.standard_normal((7, 2, 8)), rng.standard_normal((7, 2, 8))
    np.testing.assert_allclose(M.attention(q, k, v, np.full(5, 7)), M.attention(q, k, v), atol=1e-14)
    np.testing.assert_allclose(M.attention(q, k, v, np.ones(5, dtype=int)), np.broadcast_to(v[0], (5, 2, 8)),
                               atol=1e-14)


def test_block_key_limit():
    np.testing.assert_array_equal(M.block_key_limit(np.arange(12), 4, 3), [4, 4, 4, 4, 7, 7, 7, 10, 10, 10, 13, 13])


@pytest.mark.parametrize("mode", ["dual", "prefix"])
def test_block_causal_cache_is_exact(tiny_w, mode):
    """Under the block-causal mask nothing a block attends to changes after it
    is cached: the cached decoders reproduce the no-cache decoder exactly, with
    the same confidences at every step."""
    pr = synth.prompts(tiny_w.cfg, 2, 2, 12)
    ref = S.Decoder(tiny_w, pr, 24, 8, "none", mask="block_causal")
    t_ref, tr_ref = ref.generate(S.Rule(S.THRESHOLD, 0.9))
    dec = S.Decoder(tiny_w, pr, 24, 8, mode, mask="block_causal")
    t, tr = dec.generate(S.Rule(S.THRESHOLD, 0.9))
    np.testing.assert_array_equal(t, t_ref)
    assert len(tr) == len(tr_ref)
    for a, b in zip(tr, tr_ref):
        np.testing.assert_allclose(a.conf, b.conf, atol=1e-12)


def test_block_causal_prompt_ignores_answer(tiny_w):
    """A prompt row under the block-causal mask sees the prompt only: its K/V
    are those of a forward over the prompt alone."""
    pr = synth.prompts(tiny_w.cfg, 1, 1, 10)
    dec = S.Decoder(tiny_w, pr, 16, 8, "dual", mask="block_causal")
    dec.refresh()
    alone = M.forward_rows(tiny_w, pr[0], np.arange(10), None, None, skip_last_post_attn=True)
    for l in range(tiny_w.cfg.n_layers):
        np.testing.assert_allclose(dec.k_cache[0][l][:10], alone.k[l], atol=1e-12)
        np.testing.assert_allclose(dec.v_cache[0][l][:10], alone.v[l], atol=1e-12)


def test_staleness_zero_right_after_refresh(tiny_w):
    """Right after a refresh the cache is the fresh forward: every cosine is 1
    and the cached and uncached predictions are the same."""
    pr = synth.prompts(tiny_w.cfg, 0, 2, 12)
    dec = S.Decoder(tiny_w, pr, 16, 8, "dual")
    dec.refresh()
    st = S.staleness(dec, 0)
    np.testing.assert_allclose(st["k_cos"], 1.0, atol=1e-12)
    np.testing.assert_allclose(st["v_cos"], 1.0, atol=1e-12)
    assert st["agree"] == 1.0 and st["max_dconf"] < 1e-12


def test_staleness_after_commits(tiny_w):
    """After two steps inside block 0 the prefix/suffix rows of layer 0 are
    still exact (layer-0 K/V of a position depend on its own token alone), the
    deeper layers' rows have gone stale (cosine below 1, the attention mixes
    in the newly committed tokens), and everything stays a cosine."""
    pr = synth.prompts(tiny_w.cfg, 0, 1, 12)
    dec = S.Decoder(tiny_w, pr, 16, 8, "dual")
    dec.refresh()
    dec.step(0, S.Rule(S.FIXED_K, k=3))
    dec.step(0, S.Rule(S.FIXED_K, k=3))
    st = S.staleness(dec, 0)
    np.testing.assert_allclose(st["k_cos"][0], 1.0, atol=1e-12)
    np.testing.assert_allclose(st["v_cos"][0], 1.0, atol=1e-12)
    assert (st["k_cos"][1:] < 1.0 - 1e-9).all() and (st["v_cos"][1:] < 1.0 - 1e-9).all()
    assert (st["k_cos"] > 0.0).all() and 0.0 <= st["agree"] <= 1.0


@pytest.mark.parametrize("mode", ["prefix", "dual"])
def test_refresh_every_step_equals_no_cache(tiny_w, mode):
    _, t_none, tr_none = _run(tiny_w, "none", S.Rule(S.THRESHOLD, 0.9), b=2)
    _, t_c, tr_c = _run(tiny_w, mode, S.Rule(S.THRESHOLD, 0.9), b=2, refresh_interval=1)
    np.testing.assert_array_equal(t_none, t_c)
    assert len(tr_none) == len(tr_c)
    for a, b in zip(tr_none, tr_c):
        np.testing.assert_allclose(a.conf, b.conf, rtol=1e-9, atol=1e-12)


def test_refresh_interval_of_a_block_is_the_block_schedule(tiny_w):
    """A block takes at most B steps, so a refresh interval r >= B never
    refreshes inside a block: the same events as the block-boundary schedule
    (r = 0), the same tokens and confidences."""
    B = 8
    pr = synth.prompts(tiny_w.cfg, 1, 2, 16)
    runs = []
    for r in (0, B, 3 * B):
        dec = S.Decoder(tiny_w, pr, 32, B, "dual")
        runs.append([(ev[0], ev[1], ev[2].conf if ev[0] == "step" else None)
                     for ev in dec.run(S.Rule(S.FIXED_K, k=1), refresh_interval=r)])
    for other in runs[1:]:
        assert [e[:2] for e in other] == [e[:2] for e in runs[0]]
        for a, b in zip(other, runs[0]):
            if a[0] == "step":
                np.testing.assert_array_equal(a[2], b[2])


@pytest.mark.parametrize("r", [1, 2, 3])
def test_refresh_interval_counts(tiny_w, r):
    """With fixed k = 1 every block of B positions takes exactly B steps, so an
    interval r refreshes ceil(B / r) - 1 times inside each block, on top of
    the prefill and the n_blocks - 1 block-boundary refreshes; a refresh
    always comes right before the step whose in-block index is a multiple of r."""
    B, gen = 4, 12
    pr = synth.prompts(tiny_w.cfg, 2, 1, 8)
    dec = S.Decoder(tiny_w, pr, gen, B, "dual")
    evs = [e[:2] for e in dec.run(S.Rule(S.FIXED_K, k=1), refresh_interval=r)]
    n_blocks = gen // B
    expect = [("refresh", 0)]
    for j in range(n_blocks):
        for i in range(B):
            if i > 0 and i % r == 0:
                expect.append(("refresh", j))
            expect.append(("step", j))
        if j + 1 < n_blocks:
            expect.append(("refresh", j))
    assert evs == expect
    inside = -(-B // r) - 1
    assert dec.refreshes == 1 + (n_blocks - 1) + n_blocks * inside


def test_refresh_interval_two_differs_from_block_schedule_but_matches_no_cache_at_refresh_points(tiny_w):
    """Right after an in-block refresh the cache is the full forward of the
    current canvas: the step that follows computes exactly what the no-cache
    decoder computes on that canvas."""
    pr = synth.prompts(tiny_w.cfg, 3, 1, 12)
    dec = S.Decoder(tiny_w, pr, 16, 8, "dual")
    prev = None
    checked = 0
    for ev in dec.run(S.Rule(S.FIXED_K, k=1), refresh_interval=2):
        if ev[0] == "step" and prev is not None and prev[0] == "refresh":
            none = S.Decoder(tiny_w, pr, 16, 8, "none")
            none.x = ev[2].x_before.copy()
            conf, arg, _, _, _ = none.compute(ev[1])
            np.testing.assert_allclose(ev[2].conf, conf, rtol=1e-9, atol=1e-12)
            np.testing.assert_array_equal(ev[2].arg, arg)
            checked += 1
        prev = ev
    assert checked >= 4


def test_dual_cache_reads_stale_suffix(tiny_w):
    """DualCache recomputes only the block: perturbing the cached suffix changes
    the block's output, while perturbing nothing reproduces it exactly."""
    pr = synth.prompts(tiny_w.cfg, 0, 1, 16)
    dec = S.Decoder(tiny_w, pr, 32, 8, "dual")
    dec.refresh()
    c0 = dec.compute(1)[0]
    c1 = dec.compute(1)[0]
    np.testing.assert_array_equal(c0, c1)
    s = dec.block_start(1)
    for l in range(tiny_w.cfg.n_layers):
        dec.k_cache[0][l][s + 8:] *= 0.5
    c2 = dec.compute(1)[0]
    assert np.abs(c2 - c0).max() > 1e-6


def test_fixed_k_counts(tiny_w):
    for k in (1, 4):
        dec, toks, trace = _run(tiny_w, "dual", S.Rule(S.FIXED_K, k=k))
        for st in trace:
            assert st.committed[0] == min(k, int(st.eligible[0].sum()))


def test_batch_lockstep_matches_single_sequences(tiny_w):
    """Sequences are independent: a lockstep batch gives each sequence's own tokens."""
    pr = synth.prompts(tiny_w.cfg, 0, 3, 16)
    dec = S.Decoder(tiny_w, pr, 32, 8, "dual")
    toks, _ = dec.generate(S.Rule(S.THRESHOLD, 0.9))
    for i in range(3):
        d1 = S.Decoder(tiny_w, pr[i:i + 1], 32, 8, "dual")
        t1, _ = d1.generate(S.Rule(S.THRESHOLD, 0.9))
        np.testing.assert_array_equal(t1[0], toks[i])


def test_lower_tau_commits_at_least_as_many_first_step(tiny_w):
    """Fig. 5 direction (section 10): a lower threshold never commits fewer
    positions from the same confidences (checked on one step's confidences)."""
    pr = synth.prompts(tiny_w.cfg, 0, 1, 16)
    dec = S.Decoder(tiny_w, pr, 32, 32, "dual")
    dec.refresh()
    conf = dec.compute(0)[0].astype(np.float32)[0]
    e = np.ones(conf.shape[0], dtype=bool)
    counts = [S.select_threshold(conf, e, t).sum() for t in (1.0, 0.9, 0.7, 0.5)]
    assert counts == sorted(counts)


# --------------------------------------------------------------------------- teaching roofline

def test_teaching_roofline_numbers():
    g = golden("teaching_roofline.json")
    r = roofline.teaching_h100()
    assert round(r.weight_ms, 2) == g["weight_read_ms"]
    assert round(r.position_ms, 5) == g["per_position_ms"]
    assert round(r.crossover) == g["crossover_positions"]
    prefill = r.step_ms(512)
    assert round(prefill, 2) == g["prefill_512_ms"]
    assert round(prefill + 256 * r.step_ms(1)) == g["ar_prefill_plus_256_ms"]
    assert round(256 * r.step_ms(768)) == g["nocache_256_steps_of_768_ms"]
    assert round(64 * r.step_ms(768)) == g["nocache_64_steps_of_768_ms"]
    assert round(prefill + 64 * r.step_ms(32)) == g["cached_64_steps_of_32_ms"]
    assert round(prefill + 72 * r.step_ms(32)) == g["cached_72_steps_of_32_ms"]
    G, tb = g["block_G"], g["tau_bar"]
    assert round(roofline.diffusion_tokens_s(r, 10 ** 4, G, tb)) == g["diffusion_cap_tok_s"]
    assert round(1e3 / r.position_ms) == g["ar_cap_tok_s"]
    sat = min(b for b in range(1, 100) if G * (b + 1) > r.crossover)
    assert sat == g["diffusion_saturation_requests"]
    over = min(b for b in range(1, 400)
               if roofline.ar_tokens_s(r, b) >= roofline.diffusion_tokens_s(r, b, G, tb))
    assert abs(over - g["ar_overtakes_requests"]) <= 1


# --------------------------------------------------------------------------- generator

def test_splitmix64_published_vector():
    g = golden("splitmix64.json")
    assert [str(x) for x in synth.splitmix64_stream(g["seed"], 5)] == g["outputs"]
    # the vectorised counter form gives the same words
    words = synth.raw_words(g["seed"], 0, 5)
    assert [str(int(x)) for x in words] == g["outputs"]


def test_generator_slices_and_moments():
    cfg = configs.M1B
    full = synth.tensor_bf16(cfg, 0, "wq", 3)
    part = synth.tensor_bf16(cfg, 0, "wq", 3, rows=slice(100, 140))
    np.testing.assert_array_equal(full[100:140], part)
    f = synth.bf16_to_f64(full)
    assert abs(f.mean()) < 1e-4 and f.std() == pytest.approx(0.02, rel=5e-3)
    ids = synth.prompts(cfg, 0, 4, 1000)
    assert ids.min() >= 0 and ids.max() < cfg.vocab
    np.testing.assert_array_equal(synth.prompts(cfg, 0, 2, 1000, first_seq=2), ids[2:4])
    lm = synth.bf16_to_f64(synth.tensor_bf16(configs.TINY, 0, "lm_head"))
    assert lm.std() == pytest.approx(0.02 * configs.TINY.lm_scale, rel=2e-2)
