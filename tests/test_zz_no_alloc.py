"""dllm_op_attention_noalloc against dllm_op_attention (GPU, through the C ABI).

The no-alloc variant plans the key splits like dllm_op_attention and keeps its
scratch in static device storage; for every shape it accepts both must give
bit-identical outputs, on consecutive calls (the merge counters it shares
across calls must come back to zero), and a shape over its fixed scratch must
be rejected without a launch.  Collected last so that it also runs after the
other GPU tests in the same process.
"""
import numpy as np
import pytest

from cached_masked_decoding_gb300 import binding
from gpu_util import bf16_bits, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

FITS = [
    (1, 4, 64, 16, 96),     # tiny model: one block of 16 over T = 96
    (1, 4, 64, 96, 96),     # tiny refresh (all rows)
    (2, 3, 128, 32, 200),   # ragged T, two sequences
    (1, 32, 128, 32, 768),  # the 8B DualCache block
    (1, 4, 128, 40, 70),    # ragged queries and keys
]


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    binding.lib()
    return t


def _inputs(torch, b, H, hd, R, T, seed):
    rng = np.random.default_rng(seed)
    q = to_dev(torch, bf16_bits(rng.standard_normal((b, R, H, hd)).astype(np.float32)))
    k = to_dev(torch, bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32)))
    v = to_dev(torch, bf16_bits(rng.standard_normal((b, H, T, hd)).astype(np.float32)))
    return q, k, v


def test_matches_allocating_attention_on_consecutive_calls(torch):
    for i, (b, H, hd, R, T) in enumerate(FITS):
        q, k, v = _inputs(torch, b, H, hd, R, T, 100 + i)
        ref = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
        binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), ref.data_ptr(), b, H, hd, R, T)
        outs = []
        for _ in range(2):   # two calls in a row on the same stream share the static scratch
            o = torch.full((b * R, H * hd), -1, dtype=torch.int16, device="cuda")
            binding.op_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
            outs.append(o)
        torch.cuda.synchronize()
        for o in outs:
            assert torch.equal(o, ref), f"shape {(b, H, hd, R, T)} differs from dllm_op_attention"


def test_rejects_shapes_over_the_static_scratch(torch):
    b, H, hd, R, T = 1, 8, 128, 256, 768     # 6 key splits x 32 works x 64 rows x 130 floats > 1 Mi
    q, k, v = _inputs(torch, b, H, hd, R, T, 7)
    o = torch.full((b * R, H * hd), 123, dtype=torch.int16, device="cuda")
    with pytest.raises(binding.DllmError) as ei:
        binding.op_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
    assert ei.value.status == binding.EINVAL
    assert "no-alloc" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((o == 123).all()), "a rejected call must not launch"
    # the allocating entry point takes the same shape
    binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
    torch.cuda.synchronize()
