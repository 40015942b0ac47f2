"""Parity at the full 1B and 8B shapes, in the launch configuration the bench
times (the persistent one-launch DualCache step).

* 1B (16 layers, d 2048, V 32000; prompt 256, gen 128, block 32, tau 0.9):
  the whole generation under the trajectory-sync rule, every step checked
  against the oracle recomputing it on the GPU's canvas.
* 8B (32 layers, d 4096, V 126464; prompt 512, gen 256, block 32): the
  prefill refresh and the first denoise step - the K/V cache of sampled layers,
  the final hidden rows, the confidences, argmaxes and the commit of the 32
  block positions - against the oracle's refresh and block forward.  The
  oracle materialises one layer's float64 weights at a time (about 1.7 GB).
"""
import numpy as np
import pytest

from cached_masked_decoding_gb300 import binding, configs, synth
from gpu_util import torch_cuda
from oracle import model as OM
from oracle import sampler as OS
from parity import TOL, Report, conf_tol, run_synced

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    binding.lib()
    return t


class _LazyLayers:
    """Per-layer float64 weights, generated from the seeded stream on access."""

    def __init__(self, cfg, seed):
        self.cfg, self.seed = cfg, seed

    def __len__(self):
        return self.cfg.n_layers

    def __getitem__(self, l):
        return OM.LayerWeights(**{n: synth.bf16_to_f64(synth.tensor_bf16(self.cfg, self.seed, n, l))
                                  for n in synth.LAYER_TENSORS})


def _lazy_weights(cfg, seed) -> OM.Weights:
    return OM.Weights(cfg=cfg, embed=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "embed")),
                      layers=_LazyLayers(cfg, seed),
                      final_norm=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "final_norm")),
                      lm_head=synth.bf16_to_f64(synth.tensor_bf16(cfg, seed, "lm_head")))


def test_1b_generation_trajectory(torch):
    wl = configs.WORKLOADS["1b"]
    cfg = wl.model
    gm = binding.Model.from_synth(cfg, seed=wl.seed)
    pr = synth.prompts(cfg, wl.seed, wl.batch, wl.prompt_len)
    st = binding.State(gm, pr, wl.batch, wl.prompt_len, wl.gen_len, wl.block)
    st.set_persistent(True)
    dec = OS.Decoder(OM.load_weights(cfg, wl.seed), pr, wl.gen_len, wl.block, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, wl.tau), "dual")
    print("1b:", rep)
    rep.log(workload="1b", T=wl.T)
    assert rep.steps >= wl.gen_len // wl.block
    assert (st.tokens()[:, wl.prompt_len:] != cfg.mask_id).all()
    st.free()
    gm.free()


def test_1b_long_context_two_blocks(torch):
    """T = 2048 (the long-output shape: prompt 1024, gen 1024, block 32) on the
    1B-shaped model through the persistent step: the prefill refresh, block 0
    to completion, the block-boundary refresh and block 1, under the
    trajectory-sync rule.  The step's attention then splits 2048 keys 8 ways
    (256 keys, eight 32-key tiles per item), past every other tested shape."""
    cfg = configs.M1B
    wl = configs.Workload("1b_long", cfg, 1, 1024, 1024, 32)
    gm = binding.Model.from_synth(cfg, seed=wl.seed)
    pr = synth.prompts(cfg, wl.seed, wl.batch, wl.prompt_len)
    st = binding.State(gm, pr, wl.batch, wl.prompt_len, wl.gen_len, wl.block)
    st.set_persistent(True)
    dec = OS.Decoder(OM.load_weights(cfg, wl.seed), pr, wl.gen_len, wl.block, "dual")
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, wl.tau), "dual", max_blocks=2)
    print("1b T=2048:", rep)
    rep.log(workload="1b_long", T=wl.T)
    assert rep.refreshes == 2
    assert (st.tokens()[:, wl.prompt_len:wl.prompt_len + 2 * wl.block] != cfg.mask_id).all()
    st.free()
    gm.free()


@pytest.mark.parametrize("mask", ["full", "block_causal"])
def test_1b_prefix_cache_two_blocks(torch, mask):
    """PrefixCache on the 1B model (every step recomputes rows [block start,
    T)): the 128 and 96 query rows of blocks 0 and 1 take the tensor-core
    attention, whose plan cuts each query tile's 384 keys into six ranges and
    merges their partial softmax states; under the block-causal mask the rows
    of a query tile also stop at different keys.  Checked under the
    trajectory-sync rule like the DualCache trajectory."""
    wl = configs.WORKLOADS["1b"]
    cfg = wl.model
    gm = binding.Model.from_synth(cfg, seed=wl.seed)
    pr = synth.prompts(cfg, wl.seed, wl.batch, wl.prompt_len)
    st = binding.State(gm, pr, wl.batch, wl.prompt_len, wl.gen_len, wl.block)
    st.set_mask(mask)
    dec = OS.Decoder(OM.load_weights(cfg, wl.seed), pr, wl.gen_len, wl.block, "prefix", mask=mask)
    rep = run_synced(st, dec, OS.Rule(OS.THRESHOLD, wl.tau), "prefix", max_blocks=2)
    print("1b prefix:", mask, rep)
    rep.log(workload="1b_prefix", T=wl.T, mask=mask)
    assert (st.tokens()[:, wl.prompt_len:wl.prompt_len + 2 * wl.block] != cfg.mask_id).all()
    st.free()
    gm.free()


def test_8b_refresh_and_first_step(torch):
    wl = configs.WORKLOADS["8b"]
    cfg = wl.model
    gm = binding.Model.from_synth(cfg, seed=wl.seed)
    pr = synth.prompts(cfg, wl.seed, wl.batch, wl.prompt_len)
    st = binding.State(gm, pr, wl.batch, wl.prompt_len, wl.gen_len, wl.block)
    st.set_persistent(True)
    st.refresh()
    sampled = (0, cfg.n_layers // 2, cfg.n_layers - 1)
    kv_gpu = {l: st.kv(l) for l in sampled}          # after the refresh
    cnt = st.step(0, wl.tau, "dual")
    x_after, conf_g, arg_g = st.read()
    h_g = st.hidden().astype(np.float64)
    st.free()
    gm.free()

    w = _lazy_weights(cfg, wl.seed)
    dec = OS.Decoder(w, pr, wl.gen_len, wl.block, "dual")
    dec.refresh()
    for l in sampled:
        k, v = kv_gpu[l]
        for got, ref in ((k[0], dec.k_cache[0][l].transpose(1, 0, 2)), (v[0], dec.v_cache[0][l].transpose(1, 0, 2))):
            rel = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
            assert rel.max() < 1e-2, f"layer {l}: K/V row relative error {rel.max():.3e}"
    conf_o, arg_o, margin, hb, _ = dec.compute(0)
    rel = np.linalg.norm(h_g[0] - hb[0], axis=-1) / np.linalg.norm(hb[0], axis=-1)
    assert rel.max() <= 1e-2, f"final hidden relative error {rel.max():.3e}"
    err = np.abs(conf_g[0].astype(np.float64) - conf_o[0])
    assert err.max() <= conf_tol(cfg), f"max-prob error {err.max():.3e}"
    mism = np.flatnonzero(arg_g[0] != arg_o[0])
    for i in mism:
        assert margin[0, i] < TOL, f"argmax differs at position {i} with oracle margin {margin[0, i]:.3e}"
    # the commit is the threshold rule on the GPU's own confidences
    s = wl.prompt_len
    elig = np.ones(wl.block, dtype=bool)
    sel = OS.select(OS.Rule(OS.THRESHOLD, wl.tau), conf_g[0], elig)
    expect = dec.x[0].copy()
    expect[s + np.flatnonzero(sel)] = arg_g[0, np.flatnonzero(sel)]
    np.testing.assert_array_equal(x_after[0], expect)
    assert int(cnt.sum()) == int(sel.sum()) >= 1
    rep = Report()
    rep.steps, rep.refreshes, rep.decisions, rep.arg_near_ties = 1, 1, wl.block, int(mism.size)
    rep.max_conf_err, rep.max_hidden_rel = float(err.max()), float(rel.max())
    rep.log(workload="8b", T=wl.T)
    print(f"8b: max conf err {err.max():.2e}, hidden rel {rel.max():.2e}, committed {int(cnt.sum())}, "
          f"argmax near ties {mism.size}")
