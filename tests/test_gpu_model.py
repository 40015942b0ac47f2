"""Model-level parity on the GPU: the refresh K/V, one step per cache mode
layer by layer, whole trajectories under the trajectory-sync rule for every
selection rule, determinism, batching and edge cases (tiny model)."""
import numpy as np
import pytest

from cached_masked_decoding_gb300 import binding, configs, synth
from gpu_util import torch_cuda
from oracle import model as OM
from oracle import sampler as OS
from parity import conf_tol, run_loop_synced, run_synced

pytestmark = pytest.mark.gpu

CFG = configs.TINY_SPREAD


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    binding.lib()
    return t


@pytest.fixture(scope="module")
def gmodel(torch):
    m = binding.Model.from_synth(CFG, seed=0, random_norms=True)
    yield m
    m.free()


@pytest.fixture(scope="module")
def omodel():
    return OM.load_weights(CFG, 0, random_norms=True)


def test_refresh_writes_oracle_kv(gmodel, omodel):
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 0, 2, P)
    st = binding.State(gmodel, pr, 2, P, gen, B)
    st.refresh()
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    dec.refresh()
    for l in range(CFG.n_layers):
        k, v = st.kv(l)
        for i in range(2):
            ko = dec.k_cache[i][l].transpose(1, 0, 2)   # [H][T][hd]
            vo = dec.v_cache[i][l].transpose(1, 0, 2)
            for got, ref in ((k[i], ko), (v[i], vo)):
                rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
                assert rel < 1e-2, f"layer {l} seq {i}: relative K/V error {rel:.3e}"
    st.free()


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
def test_one_step_layer_by_layer(gmodel, omodel, mode):
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 0, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    st.set_trace(True)
    dec = OS.Decoder(omodel, pr, gen, B, mode)
    if mode != "none":
        st.refresh()
        dec.refresh()
    cnt = st.step(0, 0.9, mode)
    tr, R, p0 = st.trace()
    conf_o, arg_o, margin, hb, layers = dec.compute(0, keep_layers=True)
    rows = dec.rows_of(0)
    assert R == rows.size and p0 == rows[0]
    for l, ref in enumerate(layers[0]):
        got = tr[l, 0].astype(np.float64)
        rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
        assert rel.max() < 1e-2, f"{mode}: layer {l} output relative error {rel.max():.3e}"
    _, conf_g, arg_g = st.read()
    assert np.abs(conf_g[0] - conf_o[0]).max() <= conf_tol(CFG)
    assert ((arg_g[0] == arg_o[0]) | (margin[0] < 2e-3)).all()
    assert cnt.sum() >= 1
    st.free()


RULES = {
    "threshold": OS.Rule(OS.THRESHOLD, 0.9),
    "tau_gt_1": OS.Rule(OS.THRESHOLD, 1.5),
    "fixed1": OS.Rule(OS.FIXED_K, k=1),
    "fixed4": OS.Rule(OS.FIXED_K, k=4),
    "factor": OS.Rule(OS.FACTOR, factor=1.0),
    "budget": OS.Rule(OS.BUDGET),
    "schedule": OS.Rule(OS.SCHEDULE, k=6),
}


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
@pytest.mark.parametrize("rule", ["threshold", "fixed4", "factor"])
def test_trajectory_matches_oracle(gmodel, omodel, mode, rule):
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 0, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, mode)
    rep = run_synced(st, dec, RULES[rule], mode)
    print(mode, rule, rep)
    assert rep.near_ties <= max(2, rep.steps // 10)
    assert (st.tokens()[:, P:] != CFG.mask_id).all()
    st.free()


@pytest.mark.parametrize("rule", ["tau_gt_1", "fixed1", "budget", "schedule"])
def test_other_rules_dual(gmodel, omodel, rule):
    P, gen, B = 32, 32, 16
    pr = synth.prompts(CFG, 0, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    rep = run_synced(st, dec, RULES[rule], "dual")
    if rule in ("tau_gt_1", "fixed1"):
        assert rep.steps == gen       # exactly one token per step
    if rule == "schedule":
        assert rep.steps == 6 * (gen // B)   # the schedule's steps per block, exactly
    st.free()


def test_schedule_rule_is_llada_sampler_on_gpu(gmodel, omodel):
    """Page 1's LLaDA sampler: no cache, the whole answer as one block, the
    scheduled rule over 10 steps, step by step against the oracle (which the
    CPU pins tie to its own restatement of the sampler); then dllm_run's own
    countdown of k gives the same number of steps."""
    P, gen, steps = 32, 64, 10
    pr = synth.prompts(CFG, 5, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, gen)
    dec = OS.Decoder(omodel, pr, gen, gen, "none")
    rep = run_synced(st, dec, OS.Rule(OS.SCHEDULE, k=steps), "none")
    assert rep.steps == steps
    st.free()
    st = binding.State(gmodel, pr, 1, P, gen, gen)
    stats = st.run(binding.make_select(binding.SEL_SCHEDULE, k=steps), "none")
    assert stats["steps"] == steps and stats["committed"] == gen
    st.free()


@pytest.mark.parametrize("b,P,B", [(1, 32, 16), (2, 45, 16), (4, 32, 32)])
def test_persistent_step_matches_per_kernel_launches(gmodel, b, P, B):
    """The cooperative single-launch DualCache step computes what the chain of
    per-kernel launches computes (the attention key split differs, so values
    agree to float32 rounding, not bit for bit)."""
    gen = 2 * B
    pr = synth.prompts(CFG, 5, b, P)
    outs = []
    for persistent in (False, True):
        st = binding.State(gmodel, pr, b, P, gen, B)
        st.set_persistent(persistent)
        st.refresh()
        st.step(0, 0.9, "dual")
        t, c, a = st.read()
        outs.append((t, c, a, st.hidden()))
        st.free()
    (t0, c0, a0, h0), (t1, c1, a1, h1) = outs
    assert np.abs(c0 - c1).max() <= 1e-4
    np.testing.assert_array_equal(a0, a1)
    np.testing.assert_array_equal(t0, t1)
    rel = np.linalg.norm(h0 - h1, axis=-1) / np.linalg.norm(h0, axis=-1)
    assert rel.max() <= 1e-4


def test_persistent_whole_run_matches_oracle_8_blocks(gmodel, omodel):
    """A longer DualCache run through the persistent step (8 blocks, 2 sequences)."""
    P, gen, B, b = 24, 128, 16, 2
    pr = synth.prompts(CFG, 6, b, P)
    st = binding.State(gmodel, pr, b, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "dual")
    assert rep.steps >= gen // B
    st.free()


@pytest.mark.parametrize("persistent", [True, False])
def test_bf16_activation_mode(gmodel, omodel, persistent):
    """DLLM_PREC_BF16 rounds every GEMM input to bf16: the tiny model's steep
    LM head (logit sigma 10) turns those roundings into max-prob errors of up
    to ~1e-2, which is the tolerance this mode is held to.  Both the
    persistent step and the per-kernel launches (whose block attention then
    runs the bf16-only 32-key CTA) are checked."""
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 0, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    st.set_persistent(persistent)
    st.set_precision("bf16")
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    st.refresh()
    dec.refresh()
    st.step(0, 0.9, "dual")
    _, conf_g, arg_g = st.read()
    conf_o, arg_o, margin, hb, _ = dec.compute(0)
    assert np.abs(conf_g[0] - conf_o[0]).max() <= 1.5e-2
    rel = np.linalg.norm(st.hidden()[0] - hb[0], axis=-1) / np.linalg.norm(hb[0], axis=-1)
    assert rel.max() <= 1e-2
    st.free()


def test_stated_tiny_model_x8(torch):
    cfg = configs.TINY
    m = binding.Model.from_synth(cfg, seed=0)
    w = OM.load_weights(cfg, 0)
    pr = synth.prompts(cfg, 0, 1, 32)
    st = binding.State(m, pr, 1, 32, 64, 16)
    dec = OS.Decoder(w, pr, 64, 16, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "dual")
    assert rep.steps == 64            # x8 never reaches 0.9: one fallback commit per step
    st.free()
    m.free()


def test_batch_lockstep_and_ragged_prompt(gmodel, omodel):
    P, gen, B, b = 45, 48, 16, 3
    pr = synth.prompts(CFG, 3, b, P)
    st = binding.State(gmodel, pr, b, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "dual")
    assert rep.steps >= gen // B
    st.free()


def test_run_is_deterministic_and_generate_agrees(gmodel):
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 1, 2, P)
    outs = []
    for _ in range(2):
        st = binding.State(gmodel, pr, 2, P, gen, B)
        stats = st.run(binding.make_select(binding.SEL_THRESHOLD, 0.9), "dual")
        t, c, a = st.read()
        outs.append((t, c, a, stats))
        st.free()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    assert outs[0][3]["steps"] == outs[1][3]["steps"]
    assert outs[0][3]["committed"] == 2 * gen
    toks, stats = binding.generate(gmodel, pr, gen, B, 0.9, "dual")
    np.testing.assert_array_equal(toks, outs[0][0][:, P:])
    assert stats["steps"] == outs[0][3]["steps"] and stats["tau_bar"] > 0


@pytest.mark.parametrize("mask", ["full", "block_causal"])
@pytest.mark.parametrize("rule", ["threshold", "schedule"])
def test_run_ahead_takes_the_same_trajectory(gmodel, mask, rule):
    """dllm_run with run-ahead (a block's next step enqueued before the
    current step's commits are read back) decodes exactly what the loop that
    reads every step's commits first decodes: the same canvas, confidences,
    steps and refreshes (same kernels, same inputs).  The only difference is
    at most one extra launch per block: the step launched ahead of a block's
    last step, which finds no MASK and does nothing."""
    P, gen, B, b = 32, 64, 16, 2
    pr = synth.prompts(CFG, 5, b, P)
    sel = (binding.make_select(binding.SEL_THRESHOLD, 0.9) if rule == "threshold"
           else binding.make_select(binding.SEL_SCHEDULE, k=8))
    outs = []
    for ahead in (False, True):
        st = binding.State(gmodel, pr, b, P, gen, B)
        if mask != "full":
            st.set_mask(mask)
        st.set_run_ahead(ahead)
        stats = st.run(sel, "dual")
        outs.append((st.read(), stats))
        st.free()
    (t0, c0, a0), s0 = outs[0]
    (t1, c1, a1), s1 = outs[1]
    np.testing.assert_array_equal(t0, t1)
    np.testing.assert_array_equal(c0, c1)
    np.testing.assert_array_equal(a0, a1)
    assert (t1[:, P:] != CFG.mask_id).all()
    for k in ("steps", "refreshes", "committed", "fused_steps", "max_steps_per_block"):
        assert s0[k] == s1[k], k
    assert s0["tau_bar"] == s1["tau_bar"]
    n_blocks = gen // B
    assert s0["kernel_launches"] <= s1["kernel_launches"] <= s0["kernel_launches"] + n_blocks


def test_refresh_every_step_equals_no_cache_on_gpu(gmodel, omodel):
    """Invariant (iv) of the cached decoders: refreshing before every step makes
    DualCache read exactly the K/V a no-cache forward computes.  dllm_run with
    refresh interval 1 is followed step by step against the oracle's no-cache
    decoder: every step of the cached GPU run must be the no-cache step on
    the same canvas, under the trajectory-sync rule (near ties counted)."""
    P, gen, B = 32, 32, 16
    pr = synth.prompts(CFG, 2, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "none")
    rep, stats = run_loop_synced(st, dec, RULES["threshold"], "dual", refresh_interval=1, ignore_refreshes=True)
    print(rep)
    # the prefill, one refresh before every step but a block's first, and one
    # at each of the n_blocks - 1 block boundaries: as many as steps
    assert stats["refreshes"] == stats["steps"]
    st.free()


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
@pytest.mark.parametrize("rule", ["threshold", "schedule"])
def test_run_loop_matches_oracle(gmodel, omodel, mode, rule):
    """dllm_run - the block/step loop the bench times, with its refresh
    points, the skipped refresh after the last block, the lockstep batch and
    the scheduled rule's countdown - against the oracle's Algorithm 1, event
    by event (notes, section 3, Algorithm 1).  Each refresh runs fused with
    the step after it (the default)."""
    P, gen, B, b = 24, 48, 16, 2
    pr = synth.prompts(CFG, 8, b, P)
    st = binding.State(gmodel, pr, b, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, mode)
    rep, stats = run_loop_synced(st, dec, RULES[rule], mode)
    print(mode, rule, rep)
    assert stats["refreshes"] == (gen // B if mode != "none" else 0)
    assert stats["fused_steps"] == stats["refreshes"]
    assert stats["committed"] == b * gen and (st.tokens()[:, P:] != CFG.mask_id).all()
    if rule == "schedule":
        assert stats["steps"] == RULES[rule].k * (gen // B)
    st.free()


@pytest.mark.parametrize("mask", ["full", "block_causal"])
def test_run_loop_unfused_matches_oracle(gmodel, omodel, mask):
    """dllm_run with every refresh (and block-causal commit forward) run on
    its own before the step after it, as Algorithm 1 lists them: the same
    events and the same trajectory-sync bar as the fused default."""
    P, gen, B, b = 24, 48, 16, 2
    pr = synth.prompts(CFG, 8, b, P)
    st = binding.State(gmodel, pr, b, P, gen, B)
    st.set_mask(mask)
    st.set_fused_refresh(False)
    dec = OS.Decoder(omodel, pr, gen, B, "dual", mask=mask)
    rep, stats = run_loop_synced(st, dec, RULES["threshold"], "dual")
    print(mask, rep)
    assert stats["fused_steps"] == 0 and stats["refreshes"] == gen // B
    st.free()


@pytest.mark.parametrize("r", [2, 4])
def test_refresh_interval_matches_oracle(gmodel, omodel, r):
    """The refresh interval separated from the block schedule (notes, section
    11, Table 10): dllm_run(refresh_interval = r) against the oracle with the
    same interval, event by event (the in-block refreshes included)."""
    P, gen, B = 32, 48, 16
    pr = synth.prompts(CFG, 9, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    rep, stats = run_loop_synced(st, dec, OS.Rule(OS.FIXED_K, k=2), "dual", refresh_interval=r)
    print(r, rep)
    # fixed k = 2: B / 2 steps per block, a refresh before every r-th of them
    inside = -(-(B // 2) // r) - 1
    assert stats["refreshes"] == 1 + (gen // B - 1) + (gen // B) * inside
    st.free()


def test_edge_cases(gmodel, omodel):
    # one block covering the whole answer (no refresh between blocks)
    pr = synth.prompts(CFG, 4, 1, 20)
    st = binding.State(gmodel, pr, 1, 20, 32, 32)
    dec = OS.Decoder(omodel, pr, 32, 32, "dual")
    run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "dual")
    st.free()
    # no prompt at all
    st = binding.State(gmodel, np.zeros((1, 0), dtype=np.int32), 1, 0, 32, 16)
    dec = OS.Decoder(omodel, np.zeros((1, 0), dtype=np.int64), 32, 16, "prefix")
    run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "prefix")
    st.free()
    # block of one position: autoregressive-like order
    st = binding.State(gmodel, pr, 1, 20, 4, 1)
    dec = OS.Decoder(omodel, pr, 4, 1, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, 0.9), "dual")
    assert rep.steps == 4
    st.free()
    # empty answer: nothing to do
    st = binding.State(gmodel, pr, 1, 20, 0, 16)
    stats = st.run(binding.make_select(), "dual")
    assert stats["steps"] == 0 and stats["committed"] == 0
    st.free()


def test_invalid_arguments_leave_state_unchanged(gmodel):
    pr = synth.prompts(CFG, 0, 1, 8)
    with pytest.raises(binding.DllmError) as e:
        binding.State(gmodel, pr, 1, 8, 30, 16)            # gen_len % block != 0
    assert e.value.status == binding.EINVAL
    bad = pr.copy()
    bad[0, 3] = CFG.vocab                                   # MASK id in the prompt
    with pytest.raises(binding.DllmError):
        binding.State(gmodel, bad, 1, 8, 32, 16)
    st = binding.State(gmodel, pr, 1, 8, 32, 16)
    before = st.tokens()
    with pytest.raises(binding.DllmError):
        st.step(2, 0.9, "dual")                             # block index out of range
    with pytest.raises(binding.DllmError):
        st.step(0, float("nan"), "dual")
    with pytest.raises(binding.DllmError):
        st.step_ex(0, binding.make_select(binding.SEL_FIXED_K, k=0), "dual")
    np.testing.assert_array_equal(st.tokens(), before)
    st.free()


def test_weight_file_round_trip(tmp_path, gmodel, torch):
    path = str(tmp_path / "tiny.bin")
    synth.write_weight_file(path, CFG, 0, random_norms=True)
    m2 = binding.Model.load(path)
    pr = synth.prompts(CFG, 0, 1, 32)
    a, _ = binding.generate(gmodel, pr, 32, 16, 0.9, "dual")
    b, _ = binding.generate(m2, pr, 32, 16, 0.9, "dual")
    np.testing.assert_array_equal(a, b)
    m2.free()


def test_staleness_matches_oracle(gmodel, omodel):
    """The staleness diagnostic (fresh versus cached K/V and predictions) on
    the GPU against the oracle's, on the GPU's canvas after two DualCache
    steps; right after the refresh every cosine is 1."""
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 1, 2, P)
    st = binding.State(gmodel, pr, 2, P, gen, B)
    st.refresh()
    fresh = st.staleness(0)
    np.testing.assert_allclose(fresh["k_cos"], 1.0, atol=1e-6)
    np.testing.assert_allclose(fresh["v_cos"], 1.0, atol=1e-6)
    assert fresh["agree"] == 1.0 and fresh["max_dconf"] == 0.0
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    dec.refresh()
    for _ in range(2):
        st.step_ex(0, binding.make_select(binding.SEL_FIXED_K, k=3), "dual")
    dec.x = st.tokens().astype(np.int64)
    got = st.staleness(0)
    ref = OS.staleness(dec, 0)
    print({k: (got[k], ref[k]) for k in ("agree", "max_dconf")})
    np.testing.assert_allclose(got["k_cos"], ref["k_cos"], atol=2e-5)
    np.testing.assert_allclose(got["v_cos"], ref["v_cos"], atol=2e-5)
    assert abs(got["max_dconf"] - ref["max_dconf"]) <= 2 * conf_tol(CFG)
    assert abs(got["agree"] - ref["agree"]) <= 1.0 / 32 + 1e-9   # one near tie at most
    # the diagnostic leaves the canvas alone
    np.testing.assert_array_equal(st.tokens(), dec.x)
    st.free()


@pytest.mark.parametrize("mode", ["dual", "prefix", "none"])
def test_block_causal_trajectory_matches_oracle(gmodel, omodel, mode):
    """The block-causal attention mask on the GPU (per-row key limits in the
    attention kernels) against the oracle with the same mask, step by step."""
    P, gen, B = 32, 48, 16
    pr = synth.prompts(CFG, 6, 1, P)
    st = binding.State(gmodel, pr, 1, P, gen, B)
    st.set_mask("block_causal")
    dec = OS.Decoder(omodel, pr, gen, B, mode, mask="block_causal")
    rep = run_synced(st, dec, RULES["threshold"], mode)
    print(mode, rep)
    assert (st.tokens()[:, P:] != CFG.mask_id).all()
    st.free()


def test_block_causal_commit_forward_keeps_cache_exact(gmodel, omodel):
    """With the block-causal mask dllm_run replaces each block-boundary refresh
    by one forward over the finished block; the cache stays exact, so the
    DualCache run (persistent step) must decode what the oracle's no-cache
    decoder does under the same mask, step by step under the
    trajectory-sync rule.  The prefill runs with block 0's first step, and
    each commit forward in one persistent launch with the next block's first
    step (2B rows per sequence, two sequences)."""
    P, gen, B = 32, 64, 16
    pr = synth.prompts(CFG, 7, 2, P)
    st = binding.State(gmodel, pr, 2, P, gen, B)
    st.set_mask("block_causal")
    ref = OS.Decoder(omodel, pr, gen, B, "none", mask="block_causal")
    rep, stats = run_loop_synced(st, ref, RULES["threshold"], "dual", ignore_refreshes=True)
    print(rep)
    assert stats["refreshes"] == gen // B       # the prefill plus one commit forward per finished block but the last
    assert stats["fused_steps"] == gen // B
    assert (st.tokens()[:, P:] != CFG.mask_id).all()
    st.free()


@pytest.mark.parametrize("b,B", [(16, 16), (64, 16), (16, 32)])
def test_per_kernel_decode_batches(gmodel, omodel, b, B):
    """Batches over 128 block rows leave the persistent step for one launch
    per kernel: GEMMs over 256-1024 activation rows in several row tiles and
    the key-split attention over b x B query rows.  Whole generations against
    the oracle under the trajectory-sync rule."""
    P, gen = 32, 2 * B
    pr = synth.prompts(CFG, 10 + b, b, P)
    st = binding.State(gmodel, pr, b, P, gen, B)
    dec = OS.Decoder(omodel, pr, gen, B, "dual")
    rep = run_synced(st, dec, RULES["threshold"], "dual")
    print(b, B, rep)
    assert (st.tokens()[:, P:] != CFG.mask_id).all()
    st.free()
