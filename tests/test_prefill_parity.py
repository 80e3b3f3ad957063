"""Prefill GEMM (M > 8, tcgen05/TMEM) against the fp64 oracle, through the C ABI.

Bar: |y - y_ref| <= 2e-3 * sum|w x| elementwise (weights rounded once to bf16,
relative error <= 2^-9); exact where the exact result is representable; the
dequantized weights themselves bit-exact (one-hot x rows pick single weights).
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, to_dev_bits16, to_dev_u32
from _guard import guarded

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 2e-3


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


def _run(w4, x, qw, sc, qdev=None):
    import torch
    q = qdev if qdev is not None else to_dev_u32(qw)
    y = w4.w4a16_gemm(to_dev_bits16(x), q, to_dev_bits16(sc))
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("M,N,K", [(9, 16, 64), (64, 128, 128), (130, 144, 192), (257, 256, 1536),
                                   (300, 384, 2048), (1024, 128, 6144)])
def test_prefill_ragged(w4, M, N, K):
    x, qw, sc = synth.gen_w4_problem(600 + M + N, M, N, K)
    y = _run(w4, x, qw, sc)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, rel=TOL, abs_=0.0, what=f"prefill M{M} N{N} K{K}")
    assert w4.device_error() == 0


def test_prefill_all_eight_exact_zero(w4):
    M, N, K = 64, 128, 256
    qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    sc = synth.gen_scales(7, N, K)
    x = synth.gen_x(7, M, K)
    assert np.all(_run(w4, x, qw, sc) == 0.0)


def test_prefill_hand_worked(w4):
    g = json.load(open(os.path.join(GOLDEN, "hand_2x64.json")))
    rows = [g["rows"]["r0"], g["rows"]["r1"]]
    qw = np.full((16, 8), 0x88888888, dtype=np.uint32)
    sc = np.full((16, 2), 0x3F80, dtype=np.uint16)
    qw[:2] = [[int(w, 16) for w in r["words_hex"]] for r in rows]
    sc[:2] = [[int(s, 16) for s in r["steps_bf16_hex"]] for r in rows]
    k = np.arange(64)
    xs = {"ones": np.ones(64), "ramp": k.astype(float),
          "alt": np.where(k % 2 == 0, 1.0, -1.0) * (1 + (k % 4) / 4)}
    x = np.stack([synth.f64_to_bf16_bits(xs[c["x"]]) for c in g["cases"]] * 4)  # M = 12
    y = _run(w4, x, qw, sc)
    for i in range(12):
        c = g["cases"][i % 3]
        assert y[i, :2].tolist() == c["y"]
        assert np.all(y[i, 2:] == 0.0)


def test_prefill_dequant_bit_exact(w4):
    # One-hot x rows: y[m][n] is the single weight (n, k_m) as the tensor core saw
    # it, which must be bf16_rne((code - 8) * step), the gather's value.
    N, K = 256, 1536
    qw, sc = synth.gen_qweight(8, N, K), synth.gen_scales(8, N, K)
    ks = np.arange(0, K, 7)[:200]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    x[np.arange(len(ks)), ks] = 0x3F80
    y = _run(w4, x, qw, sc)
    ref, _ = oracle.embed_gather(np.arange(N), qw, sc)   # [N][K] bf16 bits
    want = synth.bf16_bits_to_f32(ref[:, ks].T)
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("N,K", [(6144, 1536), (1536, 6144)])
def test_prefill_config4_sampled(w4, N, K):
    # M = 1024 tokens; gate/up (6144 x 1536) and down (1536 x 6144); seeds 3000/3001, x 3002.
    import torch
    seed = 3000 if N == 6144 else 3001
    x = synth.gen_x(3002, 1024, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y = _run(w4, x, None, sc, qdev=qd)
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 46)]))
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(seed, N, K, rows), sc[rows])
    assert_w4_close(y[:, rows], yr, ar, rel=TOL, abs_=0.0, what=f"config4 {N}x{K}")
