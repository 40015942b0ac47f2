"""dllm_op_attention_noalloc against dllm_op_attention (GPU, through the C ABI).

The no-alloc variant plans the key splits like dllm_op_attention and keeps its
scratch in static device storage; for every shape it accepts both must give
bit-identical outputs, on consecutive calls (the merge counters it shares
across calls must come back to zero), and a shape over its fixed scratch must
be rejected without a launch.  Collected last so that it also runs after the
other GPU tests in the same process.  Callers of this variant are those that
cannot allocate device memory at call time (memory reserved up front, or
work issued where an allocation is not allowed).
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


def _planned_scratch(b, H, hd, R, T, sms):
    """The key-split plan dllm_op_attention makes for this GPU, restated:
    (merge works, scratch floats the no-alloc variant would need)."""
    wq = 2 if R <= 32 else 4
    QT = 16 * wq
    items = b * H * -(-R // QT)
    splits = 1
    if items < 2 * sms:
        splits = min(max(1, -(-T // 64)), -(-(2 * sms) // items))
    splits = min(splits, 32)
    kps = -(-(-(-T // splits)) // 64) * 64
    splits = -(-T // kps)
    return items, (items * splits * QT * (hd + 2) if splits > 1 else 0)


def test_matches_allocating_attention_on_consecutive_calls(torch):
    """Two no-alloc calls in a row per shape against dllm_op_attention; after
    the first call (which looks up the scratch's address) the calls change the
    device's free memory by nothing."""
    for i, (b, H, hd, R, T) in enumerate(FITS):
        q, k, v = _inputs(torch, b, H, hd, R, T, 100 + i)
        outs = [torch.full((b * R, H * hd), -1, dtype=torch.int16, device="cuda") for _ in range(3)]
        ref = torch.zeros((b * R, H * hd), dtype=torch.int16, device="cuda")
        binding.op_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), outs[0].data_ptr(), b, H, hd, R, T)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for o in outs[1:]:   # two calls in a row on the same stream share the static scratch
            binding.op_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), b, H, hd, R, T)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "a no-alloc call changed the device's free memory"
        assert binding.op_check() == 0
        binding.op_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), ref.data_ptr(), b, H, hd, R, T)
        torch.cuda.synchronize()
        for o in outs:
            assert torch.equal(o, ref), f"shape {(b, H, hd, R, T)} differs from dllm_op_attention"


def test_rejects_shapes_over_the_static_scratch(torch):
    """A shape whose planned key-split scratch exceeds the static array (1 Mi
    floats) is rejected without a launch; the shape is chosen from the plan
    for this GPU's SM count, so the case holds on any GPU that has one."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shape = None
    for H in range(1, 65):
        for R in (64, 128, 256, 512):
            works, floats = _planned_scratch(1, H, 128, R, 4096, sms)
            if floats > (1 << 20) and works <= 4096:
                shape = (1, H, 128, R, 4096)
                break
        if shape:
            break
    if shape is None:
        pytest.skip(f"no attention shape needs more than the static scratch on {sms} SMs")
    b, H, hd, R, T = shape
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
    assert binding.op_check() == 0
