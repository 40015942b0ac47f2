"""Kernel-level parity on the GPU through the C ABI: the seeded device
generator, the tensor-core GEMM, block attention and the select/commit rule,
each against the CPU oracle (or exact arithmetic) on the same inputs."""
import numpy as np
import pytest

from cached_masked_decoding_gb300 import binding, configs, synth
from gpu_util import bf16_bits, bits_to_f64, dev_bits, to_dev, torch_cuda
from oracle import model as OM
from oracle import sampler as OS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    binding.lib()
    return t


# --------------------------------------------------------------------------- generator

@pytest.mark.parametrize("name,layer", [("embed", 0), ("wq", 1), ("wd", 0), ("lm_head", 0), ("attn_norm", 1)])
def test_device_generator_matches_numpy(torch, name, layer):
    cfg = configs.TINY_SPREAD
    n = int(np.prod(synth.tensor_shape(cfg, name)))
    buf = torch.empty(n, dtype=torch.int16, device="cuda")
    synth.device_fill_tensor(buf.data_ptr(), cfg, 7, name, layer, random_norms=True)
    torch.cuda.synchronize()
    ref = synth.tensor_bf16(cfg, 7, name, layer, random_norms=True).reshape(-1)
    np.testing.assert_array_equal(dev_bits(torch, buf), ref)


def test_device_prompts_match_numpy(torch):
    cfg = configs.M8B
    buf = torch.empty(3 * 512, dtype=torch.int32, device="cuda")
    synth.device_fill_prompts(buf.data_ptr(), cfg, 0, 3, 512)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(buf.cpu().numpy().reshape(3, 512), synth.prompts(cfg, 0, 3, 512))


# --------------------------------------------------------------------------- GEMM

GEMM_SHAPES = [
    (128, 32, 64),        # one tile, one chunk
    (256, 16, 256),       # N below the tile width
    (384, 32, 4096),      # stream-K: tiles cut between CTAs
    (200, 40, 320),       # ragged M, N, K
    (12288, 32, 4096),    # the 8B QKV projection at one block
    (4096, 64, 12288),    # the 8B down projection, two sequences
    (1024, 300, 512),     # several activation tiles (BN = 256)
    (640, 96, 1024),      # BN = 128
    (2048, 2048, 256),    # the compute-bound batch shape
    (12288, 768, 256),    # refresh-shaped: 576 tiles, three whole waves + a stream-K remainder
    (2432, 1024, 128),    # exactly one whole wave of 152 tiles (split), no remainder
]


@pytest.mark.parametrize("split", [False, True], ids=["bf16", "split"])
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_matches_fp64(torch, M, N, K, split):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    Wb = bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    xf = rng.standard_normal((N, K)).astype(np.float32)
    Xb = bf16_bits(xf)
    Xl = bf16_bits(xf - bits_to_f64(Xb).astype(np.float32))
    W, X, XL = to_dev(torch, Wb), to_dev(torch, Xb), to_dev(torch, Xl)
    Y = torch.zeros((N, M), dtype=torch.float32, device="cuda")
    binding.op_gemm(W.data_ptr(), X.data_ptr(), Y.data_ptr(), M, N, K, X_lo_ptr=XL.data_ptr() if split else 0)
    torch.cuda.synchronize()
    y = Y.cpu().numpy().astype(np.float64)
    w64, x64 = bits_to_f64(Wb), bits_to_f64(Xb)
    if split:
        x64 = x64 + bits_to_f64(Xl)
        # the pair carries the float32 input to ~2^-16 relative
        assert np.abs(x64 - xf).max() <= 2.0 ** -15 * np.abs(xf).max()
    ref = x64 @ w64.T
    bound = np.abs(x64) @ np.abs(w64).T          # sum_k |x_k w_k|
    err = np.abs(y - ref)
    assert (err <= 2e-6 * bound + 1e-6).all(), f"max err {err.max():.3e}, worst ratio {(err / (bound + 1e-30)).max():.3e}"
    # deterministic: a second launch gives the same bits
    Y2 = torch.zeros_like(Y)
    binding.op_gemm(W.data_ptr(), X.data_ptr(), Y2.data_ptr(), M, N, K, X_lo_ptr=XL.data_ptr() if split else 0)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)


# --------------------------------------------------------------------------- attention

ATTN_SHAPES = [
    (1, 4, 64, 16, 96),     # tiny model: one block of 16 over T = 96
    (1, 4, 64, 96, 96),     # tiny refresh (all rows)
    (2, 3, 128, 32, 200),   # ragged T, two sequences
    (1, 32, 128, 32, 768),  # the 8B DualCache step (12 key splits)
    (1, 8, 128, 256, 768),  # PrefixCache-sized query set
    (1, 4, 128, 40, 70),    # ragged queries and keys
]


@pytest.mark.parametrize("b,H,hd,R,T", ATTN_SHAPES)
def test_attention_matches_oracle(torch, b, H, hd, R, T):
    rng = np.random.default_rng(b + H + hd + R + T)
    qb = bf16_bits(rng.standard_normal((b, R, H, hd)).astype(np.float32))
    kb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    vb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    q, k, v = to_dev(torch, qb), to_dev(torch, kb), to_dev(torch, vb)
    o = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
    binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
    torch.cuda.synchronize()
    got = bits_to_f64(dev_bits(torch, o)).reshape(b, R, H, hd)
    for s in range(b):
        ref = OM.attention(bits_to_f64(qb[s]), bits_to_f64(kb[s]).transpose(1, 0, 2),
                           bits_to_f64(vb[s]).transpose(1, 0, 2))
        vmax = np.abs(bits_to_f64(vb[s])).max()
        err = np.abs(got[s] - ref)
        # P rounded to bf16 (2^-8 of sum p|v|) plus the bf16 output (2^-9 |o|)
        assert (err <= 6e-3 * vmax + 4e-3 * np.abs(ref)).all(), f"seq {s}: max err {err.max():.3e}"
    o2 = torch.zeros_like(o)
    binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), b, H, hd, R, T)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)


TC_ATTN_SHAPES = [
    (1, 4, 64, 96, 96),      # tiny refresh: one 128-query tile, 32 rows past R
    (1, 8, 128, 768, 768),   # 8B refresh-sized: 6 query tiles, 12 key tiles
    (2, 3, 128, 200, 200),   # ragged R and T (T not a multiple of 64), two sequences
    (1, 4, 128, 130, 70),    # a second query tile with 2 rows; 2 key tiles, the last with 6 keys
    (3, 2, 64, 65, 1000),    # smallest row count that takes this kernel; long keys
    (1, 1, 64, 70, 1),       # a single key
    (3, 1, 128, 65, 63),     # fewer keys than one tile; three sequences of 65 rows
    (2, 2, 64, 129, 129),    # one row and one key past a tile boundary
    (1, 40, 128, 512, 512),  # 160 query tiles: planned as one whole wave of 152 and 8 tiles in key splits
]


# None: the library's own split plan; 1: every query tile walks all keys in
# one CTA; 3: three key ranges merged by the last to finish (fewer when T is short)
@pytest.mark.parametrize("splits", [None, 1, 3])
@pytest.mark.parametrize("b,H,hd,R,T", TC_ATTN_SHAPES)
def test_tensor_core_attention_matches_oracle(torch, b, H, hd, R, T, splits):
    rng = np.random.default_rng(7 * b + H + hd + R + T)
    qb = bf16_bits(rng.standard_normal((b, R, H, hd)).astype(np.float32))
    kb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    vb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    q, k, v = to_dev(torch, qb), to_dev(torch, kb), to_dev(torch, vb)
    o = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
    binding.op_attention_tc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T, splits=splits)
    torch.cuda.synchronize()
    got = bits_to_f64(dev_bits(torch, o)).reshape(b, R, H, hd)
    for s in range(b):
        ref = OM.attention(bits_to_f64(qb[s]), bits_to_f64(kb[s]).transpose(1, 0, 2),
                           bits_to_f64(vb[s]).transpose(1, 0, 2))
        vmax = np.abs(bits_to_f64(vb[s])).max()
        err = np.abs(got[s] - ref)
        # P rounded to bf16 (2^-8 of sum p|v|) plus the bf16 output (2^-9 |o|)
        assert (err <= 6e-3 * vmax + 4e-3 * np.abs(ref)).all(), f"seq {s}: max err {err.max():.3e}"
    o2 = torch.zeros_like(o)
    binding.op_attention_tc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), b, H, hd, R, T, splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert binding.op_check() == 0


@pytest.mark.parametrize("splits", [1, 2, 8])
def test_tensor_core_attention_peaked_rows(torch, splits):
    # rows whose max moves by far more than 8 (base 2) between key tiles:
    # the running output is rescaled in tensor memory (one or two key
    # ranges), or the ranges' maxima differ widely in the merge (eight)
    b, H, hd, R, T = 1, 2, 128, 128, 512
    rng = np.random.default_rng(11)
    qf = rng.standard_normal((b, R, H, hd)).astype(np.float32)
    kf = rng.standard_normal((b, H, T, hd)).astype(np.float32)
    kf[:, :, 300:] *= 4.0           # later keys score much higher
    qb, kb = bf16_bits(qf), bf16_bits(kf)
    vb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    q, k, v = to_dev(torch, qb), to_dev(torch, kb), to_dev(torch, vb)
    o = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
    binding.op_attention_tc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T, splits=splits)
    torch.cuda.synchronize()
    got = bits_to_f64(dev_bits(torch, o)).reshape(R, H, hd)
    ref = OM.attention(bits_to_f64(qb[0]), bits_to_f64(kb[0]).transpose(1, 0, 2), bits_to_f64(vb[0]).transpose(1, 0, 2))
    vmax = np.abs(bits_to_f64(vb[0])).max()
    err = np.abs(got - ref)
    assert (err <= 6e-3 * vmax + 4e-3 * np.abs(ref)).all(), f"max err {err.max():.3e}"


def test_attention_identical_keys_is_mean_of_values(torch):
    b, H, hd, R, T = 1, 2, 128, 32, 300
    rng = np.random.default_rng(5)
    qb = bf16_bits(rng.standard_normal((b, R, H, hd)).astype(np.float32))
    krow = rng.standard_normal((1, H, 1, hd)).astype(np.float32)
    kb = bf16_bits(np.broadcast_to(krow, (b, H, T, hd)))
    vb = bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32))
    q, k, v = to_dev(torch, qb), to_dev(torch, kb), to_dev(torch, vb)
    o = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
    binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
    torch.cuda.synchronize()
    got = bits_to_f64(dev_bits(torch, o)).reshape(R, H, hd)
    mean = bits_to_f64(vb[0]).mean(axis=1)        # [H][hd]
    np.testing.assert_allclose(got, np.broadcast_to(mean, (R, H, hd)), atol=4e-3)


# --------------------------------------------------------------------------- select / commit

def _select_case(rng, b, B, T, blk, mask_id, near):
    conf = rng.uniform(0.0, 1.0, size=(b, B)).astype(np.float32)
    # ties, exact thresholds and near-threshold values
    conf[:, 1] = conf[:, 0]
    conf[:, 2] = np.float32(near)
    conf[:, 3] = np.nextafter(np.float32(near), np.float32(0))
    arg = rng.integers(0, mask_id, size=(b, B)).astype(np.int32)
    x = rng.integers(0, mask_id, size=(b, T)).astype(np.int32)
    elig = rng.random((b, B)) < 0.7
    elig[0] = True
    if b > 2:
        elig[2] = False           # a finished sequence commits nothing
    x[:, blk:blk + B] = np.where(elig, mask_id, x[:, blk:blk + B])
    return conf, arg, x


RULES = [
    ("threshold", OS.Rule(OS.THRESHOLD, 0.9), binding.make_select(binding.SEL_THRESHOLD, 0.9)),
    ("threshold_hi", OS.Rule(OS.THRESHOLD, 0.999), binding.make_select(binding.SEL_THRESHOLD, 0.999)),
    ("tau_gt_1", OS.Rule(OS.THRESHOLD, 1.5), binding.make_select(binding.SEL_THRESHOLD, 1.5)),
    ("fixed1", OS.Rule(OS.FIXED_K, k=1), binding.make_select(binding.SEL_FIXED_K, k=1)),
    ("fixed4", OS.Rule(OS.FIXED_K, k=4), binding.make_select(binding.SEL_FIXED_K, k=4)),
    ("factor1", OS.Rule(OS.FACTOR, factor=1.0), binding.make_select(binding.SEL_FACTOR, factor=1.0)),
    ("factor3", OS.Rule(OS.FACTOR, factor=3.0), binding.make_select(binding.SEL_FACTOR, factor=3.0)),
    ("budget", OS.Rule(OS.BUDGET), binding.make_select(binding.SEL_BUDGET)),
]


@pytest.mark.parametrize("rule_name,orule,grule", RULES, ids=[r[0] for r in RULES])
@pytest.mark.parametrize("B", [16, 32, 64, 256])
def test_select_commit_bit_exact(torch, rule_name, orule, grule, B):
    rng = np.random.default_rng(B)
    b, mask_id = 4, 1024
    T = B + 40
    blk = 17 if T - B > 17 else 0
    for trial in range(5):
        conf, arg, x = _select_case(rng, b, B, T, blk, mask_id, 0.9 if trial % 2 == 0 else 0.95)
        if trial == 4:
            conf[:] = np.float32(0.5)          # all tied
        c_d, a_d, x_d = to_dev(torch, conf), to_dev(torch, arg), to_dev(torch, x)
        cnt = torch.zeros(b, dtype=torch.int32, device="cuda")
        binding.op_select_commit(c_d.data_ptr(), a_d.data_ptr(), x_d.data_ptr(), b, T, blk, B, mask_id, grule,
                                 cnt.data_ptr())
        torch.cuda.synchronize()
        x_ref = x.copy()
        cnt_ref = np.zeros(b, dtype=np.int32)
        for i in range(b):
            elig = x[i, blk:blk + B] == mask_id
            sel = OS.select(orule, conf[i], elig)
            x_ref[i, blk + np.flatnonzero(sel)] = arg[i, np.flatnonzero(sel)]
            cnt_ref[i] = sel.sum()
        np.testing.assert_array_equal(x_d.cpu().numpy(), x_ref)
        np.testing.assert_array_equal(cnt.cpu().numpy(), cnt_ref)
