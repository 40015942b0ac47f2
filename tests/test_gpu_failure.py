"""Failure detection on the device without a fault (GPU, through the C ABI).

Every wait in the library's kernels is bounded in time; on expiry the waiting
kernel records a site code in an error word, stops waiting and returns, and
the host reports DLLM_ETIMEOUT.  These tests make such a wait run out on
purpose - a flag that nothing raises, a one-millisecond limit, nothing else in
flight - and check the status, that the error word is cleared, and that the
next calls run normally.
"""
import numpy as np
import pytest

from cached_masked_decoding_gb300 import binding
from gpu_util import bf16_bits, bits_to_f64, to_dev, torch_cuda

pytestmark = pytest.mark.gpu

ERR_PROBE = 901


@pytest.fixture(scope="module")
def torch():
    t = torch_cuda()
    binding.lib()
    return t


def test_bounded_wait_gives_up_and_the_next_call_is_clean(torch):
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    # nothing raises the flag: the wait gives up after 1 ms
    assert binding.op_wait_probe(flag.data_ptr(), 1, 1000) == binding.ETIMEOUT
    assert "bounded wait" in binding.lib().dllm_last_error().decode()
    # the probe's check cleared the error word: the next check is clean
    assert binding.op_check() == 0
    # a raised flag is seen at once
    flag.fill_(3)
    torch.cuda.synchronize()
    assert binding.op_wait_probe(flag.data_ptr(), 3, 1000) == binding.OK
    assert binding.op_wait_probe(flag.data_ptr(), 2, 1000) == binding.OK
    # and again a timeout, then a normal kernel-level call gives correct results
    assert binding.op_wait_probe(flag.data_ptr(), 4, 2000) == binding.ETIMEOUT
    rng = np.random.default_rng(0)
    M, N, K = 256, 32, 512
    w = bf16_bits(rng.standard_normal((M, K)).astype(np.float32) * 0.05)
    x = bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    w_d, x_d = to_dev(torch, w), to_dev(torch, x)
    y = torch.zeros((N, M), dtype=torch.float32, device="cuda")
    binding.op_gemm(w_d.data_ptr(), x_d.data_ptr(), y.data_ptr(), M, N, K)
    assert binding.op_check() == 0
    ref = bits_to_f64(x) @ bits_to_f64(w).T
    np.testing.assert_allclose(y.cpu().numpy(), ref, rtol=1e-4, atol=1e-4)


def test_probe_rejects_bad_arguments(torch):
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    for limit in (0, -5, 2000001):
        assert binding.op_wait_probe(flag.data_ptr(), 1, limit) == binding.EINVAL
    assert binding.op_wait_probe(0, 1, 100) == binding.EINVAL
    assert binding.op_wait_probe(flag.data_ptr() + 2, 1, 100) == binding.EINVAL
