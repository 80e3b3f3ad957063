"""The allocation-free argmax GEMV against the regular one and the oracle (GPU).

w4a16_gemv_argmax_noalloc serves callers that cannot allocate device memory (a
plug-in whose host process owns every device allocation, a real-time decode
loop that must not reach the driver's allocator after start-up); its scratch is
a fixed array in the library's device image. It must give the same logits
(within the GEMV tolerance) and the same greedy indices as w4a16_gemv_argmax,
on consecutive calls that share that array; the logits must also meet the
oracle's bound and the index must be the oracle's, and once the first call has
done its per-device set-up, further calls must leave the device's free memory
unchanged. This file is collected last so a stop at the first failure has
already run everything else.
"""
import ctypes

import numpy as np
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
    return guarded(w4)


@pytest.mark.parametrize("M,N,K", [(1, 20000, 1536), (2, 3001, 2048), (8, 5000, 1536)])
def test_noalloc_matches_regular_on_two_calls(w4, M, N, K):
    import torch
    x, qw, sc = synth.gen_w4_problem(4000 + M, M, N, K)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    y_ref, a_ref = w4.w4a16_gemv_argmax(xd, qd, sd)
    torch.cuda.synchronize()
    y_or, absy = oracle.gemm(x, qw, sc)
    y_ref, a_ref = y_ref.cpu().numpy(), a_ref.cpu().numpy()
    for _ in range(2):
        y, a = w4.w4a16_gemv_argmax_noalloc(xd, qd, sd)
        torch.cuda.synchronize()
        y, a = y.cpu().numpy(), a.cpu().numpy()
        assert_w4_close(y, y_ref.astype(np.float64), absy, what="noalloc vs regular")
        assert np.array_equal(a, a_ref)
        # and against the oracle: the logits within the bound, the index exact
        assert_w4_close(y, y_or, absy, what="noalloc vs oracle")
        for m in range(M):
            idx, gap = oracle.argmax(y_or[m])
            assert gap > 2 * (1e-4 * absy[m, idx] + 1e-6), "ambiguous seed"
            assert a[m] == idx, (m, a[m], idx)


def test_noalloc_calls_leave_free_memory_unchanged(w4):
    """After the first call (the per-device set-up), calls through the C ABI with
    caller-owned buffers change the device's free memory by nothing."""
    import torch
    M, N, K = 1, 40000, 1536
    x, qw, sc = synth.gen_w4_problem(4050, M, N, K)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    a = torch.empty((M,), dtype=torch.int32, device="cuda")
    P = ctypes.c_void_p
    lib = w4._lib

    def call():
        rc = lib.w4a16_gemv_argmax_noalloc(P(y.data_ptr()), P(a.data_ptr()), P(xd.data_ptr()), P(qd.data_ptr()),
                                           P(sd.data_ptr()), M, N, K, 32, None)
        assert rc == 0

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    y_or, _ = oracle.gemm(x, qw, sc)
    assert int(a.item()) == oracle.argmax(y_or[0])[0]


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
