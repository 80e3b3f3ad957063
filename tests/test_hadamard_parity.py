"""GPU parity of w4a16_gemv_hadamard (Hadamard-rotated weights) against the fp64
oracle's (x H) W'^T, through the C ABI.

Source: "fastgemma-gemma-4-E2B" model card, "What is in the file" (every linear
weight rotated along K with a runtime fast Walsh-Hadamard transform of the
activation; FFN and LM head int4 with group 256). Bar: the decode GEMV's
|y - y_ref| <= 1e-4 * sum|w' (xH)| + 1e-6 (x H is carried as two bf16 parts,
relative 2^-18); argmax identical to the oracle's.
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
    w4.init()
    return guarded(w4)


@pytest.mark.parametrize("M,N,K,b,group", [(1, 2560, 1536, 512, 32), (1, 1536, 6144, 256, 256),
                                           (2, 300, 2048, 128, 64), (3, 500, 1024, 32, 32),
                                           (4, 2560, 1536, 512, 256), (1, 70, 512, 2, 32),
                                           (1, 33, 4096, 4096, 512), (2, 1536, 12288, 512, 256),
                                           # fused into the decode kernel's staging (M = 1, blocks of
                                           # 256 / 512): many blocks per warp, one block, ragged N
                                           (1, 1536, 12288, 512, 256), (1, 48, 256, 256, 32),
                                           (1, 4000, 2048, 256, 64),
                                           # the shared-memory slot form (group 32, K % 768 == 0):
                                           # the rotated sweep's long shapes, a shorter last CTA
                                           (1, 24576, 1536, 512, 32), (1, 1536, 12288, 512, 32),
                                           (1, 12288, 1536, 256, 32), (1, 1536, 6144, 512, 32),
                                           (1, 2576, 1536, 256, 32)])
def test_rotated_gemv_matches_oracle(w4, M, N, K, b, group):
    import torch
    x = synth.gen_x(900 + M + b, M, K)
    qw = synth.gen_qweight(900 + N, N, K)
    sc = synth.gen_scales(900 + N, N, K, group)
    y = w4.w4a16_gemv_hadamard(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), b, group=group)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm_hadamard(x, qw, sc, b, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"hadamard M{M} N{N} K{K} b{b} g{group}")


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_rotated_lm_head_argmax(w4, M):
    """The vocabulary-projection forms (persistent kernels; at M = 2..4 the pair
    rows take the M <= 8 one) with the LM head's group 256 and the fused greedy
    pick."""
    import torch
    N, K, b, group = 80000, 1536, 512, 256
    x = synth.gen_x(950 + M, M, K)
    qw = synth.gen_qweight(951, N, K)
    sc = synth.gen_scales(951, N, K, group)
    q = synth.gen_qweight_torch(951, N, K, torch.device("cuda"))
    y, a = w4.w4a16_gemv_hadamard(to_dev_bits16(x), q, to_dev_bits16(sc), b, group=group, argmax=True)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm_hadamard(x, qw, sc, b, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"rotated LM head M{M}")
    for m in range(M):
        idx, gap = oracle.argmax(yr[m])
        assert gap > 2 * (1e-4 * ar[m, idx] + 1e-6), "ambiguous seed"
        assert int(a.cpu().numpy()[m]) == idx


def test_fused_rotation_matches_a_prerotated_activation(w4):
    """The fused call against the oracle's product of the same weights with an
    activation rotated separately (oracle.hadamard, then the fp64 product)."""
    import torch
    M, N, K, b = 1, 512, 2048, 256
    x = synth.gen_x(960, M, K)
    qw = synth.gen_qweight(961, N, K)
    sc = synth.gen_scales(961, N, K)
    y = w4.w4a16_gemv_hadamard(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), b).cpu().numpy()
    xr = oracle.hadamard(x, b)
    yr, ar = oracle.gemm_xf64(xr, qw, sc)
    assert_w4_close(y, yr, ar, what="fused vs pre-rotated")


def test_rejects_unsupported(w4):
    import torch
    K = 1024
    x = torch.zeros((5, K), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((64, K // 8), dtype=torch.int32, device="cuda")
    s = torch.zeros((64, K // 32), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((5, 64), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    f = w4._lib.w4a16_gemv_hadamard
    assert f(P(y.data_ptr()), None, P(x.data_ptr()), P(q.data_ptr()), P(s.data_ptr()), 5, 64, K, 32, 256, None) == 2
    assert f(P(y.data_ptr()), None, P(x.data_ptr()), P(q.data_ptr()), P(s.data_ptr()), 1, 64, K, 32, 96, None) == 2
    assert f(P(y.data_ptr()), None, P(x.data_ptr()), P(q.data_ptr()), P(s.data_ptr()), 1, 64, K, 32, 2048, None) == 1
