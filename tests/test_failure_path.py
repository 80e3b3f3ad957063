"""The failure path of the bounded waits, exercised without a GPU fault.

Every kernel of the library that waits on a barrier bounds the wait; when it
runs out, the kernel sets a bit of the device error word and returns. The
self-test entry point launches a kernel whose barrier nothing arrives at: the
wait must give up, report bit 2 through w4_device_error, leave the word clear
after the read, and leave the context able to run an ordinary call whose result
still matches the oracle.
"""
import time

import pytest

import oracle
import synth
from _util import assert_w4_close, to_dev_bits16, to_dev_u32
from _guard import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


def test_wait_timeout_sets_error_bit_and_context_survives(w4):
    import torch
    torch.cuda.synchronize()
    assert w4.device_error() == 0
    t0 = time.perf_counter()
    w4.selftest_wait_timeout()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, elapsed  # the wait gave up on its own
    assert w4.device_error() == 4
    assert w4.device_error() == 0  # read-and-clear

    M, N, K = 1, 512, 1024
    x, qw, sc = synth.gen_x(830, M, K), synth.gen_qweight(830, N, K), synth.gen_scales(830, N, K, 32)
    y = w4.w4a16_gemv(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc))
    torch.cuda.synchronize()
    yr, ar = oracle.gemm(x, qw, sc, 32)
    assert_w4_close(y.cpu().numpy(), yr, ar, what="GEMV after the self-test")
    assert w4.device_error() == 0


def test_wait_timeout_on_a_side_stream(w4):
    import torch
    s = torch.cuda.Stream()
    w4.selftest_wait_timeout(s)
    s.synchronize()
    assert w4.device_error() == 4
