"""Pins of the oracle's Hadamard rotation (no GPU).

Source: "fastgemma-gemma-4-E2B" model card, "What is in the file": every linear
weight is Hadamard-rotated along K; H is orthogonal, so W' = W H^T with a
runtime fast Walsh-Hadamard transform of the activation is mathematically
identical. Reading: H = blockdiag(H_b) with the normalised Sylvester matrix
H_b[i][j] = (-1)^popcount(i & j) / sqrt(b) (symmetric, orthogonal), so the
rotated product is y = (x H) W'^T = x W^T.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _val(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_block_of_two_closed_form():
    x = synth.f64_to_bf16_bits(np.array([[1.5, -0.25, 3.0, 2.0]]))
    r = oracle.hadamard(x, 2)
    s = 1.0 / math.sqrt(2.0)
    np.testing.assert_allclose(r[0], [(1.5 - 0.25) * s, (1.5 + 0.25) * s, 5.0 * s, 1.0 * s], rtol=1e-15)


@pytest.mark.parametrize("b", [4, 16, 128, 512])
def test_matches_library_hadamard(b):
    linalg = pytest.importorskip("scipy.linalg")
    M, K = 3, 1024
    x = synth.gen_x(40 + b, M, K)
    r = oracle.hadamard(x, b)
    Hb = linalg.hadamard(b) / math.sqrt(b)
    ref = np.concatenate([_val(x)[:, i:i + b] @ Hb for i in range(0, K, b)], axis=1)
    np.testing.assert_allclose(r, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("b", [8, 64, 256])
def test_rotation_is_symmetric_orthogonal_involution(b):
    """Rows of H from unit vectors: H = H^T and H H = I; norms are kept (Parseval)."""
    E = synth.f64_to_bf16_bits(np.eye(b))
    H = oracle.hadamard(E, b)
    np.testing.assert_allclose(H, H.T, atol=1e-15)
    np.testing.assert_allclose(H @ H, np.eye(b), atol=1e-13)
    x = synth.gen_x(50 + b, 4, 4 * b)
    r = oracle.hadamard(x, b)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(_val(x), axis=1), rtol=1e-13)


@pytest.mark.parametrize("b,group", [(32, 32), (128, 64), (512, 256)])
def test_rotated_product_equals_the_unrotated_one(b, group):
    """(x H) W'^T == x W^T with W = W' H (dense fp64, scipy's H): the page's
    'mathematically identical', through the oracle's rotated GEMV."""
    linalg = pytest.importorskip("scipy.linalg")
    M, N, K = 2, 6, 1024
    x = synth.gen_x(60 + b, M, K)
    qw = synth.gen_qweight(60 + b, N, K)
    sc = synth.gen_scales(60 + b, N, K, group)
    y, absy = oracle.gemm_hadamard(x, qw, sc, b, group)
    Wp = oracle.dequant(qw, sc, group)
    HK = np.kron(np.eye(K // b), linalg.hadamard(b) / math.sqrt(b))
    W = Wp @ HK
    np.testing.assert_allclose(y, _val(x) @ W.T, rtol=1e-11, atol=1e-11)
    xr = _val(x) @ HK
    np.testing.assert_allclose(absy, np.abs(xr[:, None, :] * Wp[None, :, :]).sum(axis=2), rtol=1e-12)
