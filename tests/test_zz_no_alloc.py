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
    # Checked on the host before any launch: the pointers are never touched.
    A = ctypes.c_void_p(1 << 20)
    rc = w4._lib.w4a16_gemv_argmax_noalloc(A, A, A, A, A, 8, 1 << 22, 256, 32, None)
    assert rc == 2
