"""The allocation-free argmax GEMV against the regular one (GPU).

w4a16_gemv_argmax_noalloc serves callers that cannot allocate device memory;
its scratch is a fixed array in the library's device image. It must give the
same logits (within the GEMV tolerance) and the same greedy indices as
w4a16_gemv_argmax, on consecutive calls that share that array. This file is
collected last so a stop at the first failure has already run everything else.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, to_dev_bits16, to_dev_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    return w4


@pytest.mark.parametrize("M,N,K", [(1, 20000, 1536), (2, 3001, 2048), (8, 5000, 1536)])
def test_noalloc_matches_regular_on_two_calls(w4, M, N, K):
    import torch
    x, qw, sc = synth.gen_w4_problem(4000 + M, M, N, K)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    y_ref, a_ref = w4.w4a16_gemv_argmax(xd, qd, sd)
    torch.cuda.synchronize()
    _, absy = oracle.gemm(x, qw, sc)
    y_ref, a_ref = y_ref.cpu().numpy(), a_ref.cpu().numpy()
    for _ in range(2):
        y, a = w4.w4a16_gemv_argmax_noalloc(xd, qd, sd)
        torch.cuda.synchronize()
        y, a = y.cpu().numpy(), a.cpu().numpy()
        assert_w4_close(y, y_ref.astype(np.float64), absy, what="noalloc vs regular")
        assert np.array_equal(a, a_ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(w4):
    """A call whose plan needs more argmax keys than the fixed scratch holds is
    refused on the host. K = 160 (not a multiple of 128) keeps the large-N forms
    out, so 8 x-rows over 2^22 rows need 8 x 32768 keys against 32768. The
    buffers are real (zeroed), so no plan could make the call touch an invalid
    address."""
    import torch
    M, N, K = 8, 1 << 22, 160
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    a = torch.zeros((M,), dtype=torch.int32, device="cuda")
    x = torch.zeros((M, K), dtype=torch.int16, device="cuda")
    q = torch.zeros((N, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((N, K // 32), dtype=torch.int16, device="cuda")
    P = ctypes.c_void_p
    rc = w4._lib.w4a16_gemv_argmax_noalloc(P(y.data_ptr()), P(a.data_ptr()), P(x.data_ptr()), P(q.data_ptr()),
                                           P(sc.data_ptr()), M, N, K, 32, None)
    torch.cuda.synchronize()
    assert rc == 2
