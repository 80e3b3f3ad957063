"""The vocabulary-sized decode GEMV for 2..8 x-rows with the weights landed in
shared-memory slots by tensor copies (group 32, K a multiple of 768, at least
two 16-row blocks per warp of a full wave), against the fp64 oracle through
the C ABI.

Covers x-row counts 2..8 (zero B columns beyond M), one to four six-tile units
per row (K = 768 .. 3072), a last row block that only some warps reach, x
staged as fp16 when every value is exact there and a thread holds few chunks,
else as bf16 (values beyond fp16's exact range; long K), and the fused greedy
pick per x-row. Bar: |y - y_ref| <= 1e-4 * sum|w x| + 1e-6 elementwise on
sampled rows, the pick exact against the oracle's pick over every row, run to
run bitwise identical results.

Source: "fastgemma-gemma-4-E2B" (batch-8 serving: 8 sequences share one read
of the weights) and "Gemma 4 E2B on a 4 GB GPU with pure PyTorch", Step 2 (the
tied 4-bit embedding read once per token as the output layer).
"""
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


def _rows(N):
    return np.unique(np.concatenate([[0, 1, 15, 16, N - 17, N - 1], np.arange(29, N, 1031)]))


def _check(w4, x, seed, N, K, what):
    import torch
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y = w4.w4a16_gemv(to_dev_bits16(x), qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    rows = _rows(N)
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(seed, N, K, rows), sc[rows])
    assert_w4_close(y[:, rows], yr, ar, what=what)
    return y


# (N, K): one unit per row is not served (K >= 1536 keeps two); 2..4 units per
# row; N not a multiple of the wave's warps (the last row blocks reach only
# some warps).
SHAPES = [(80000, 1536), (131072, 2304), (98304, 3072), (77840, 1536)]


@pytest.mark.parametrize("M", [2, 3, 5, 8])
@pytest.mark.parametrize("N,K", SHAPES)
def test_slots8_shapes(w4, M, N, K):
    seed = 5000 + N % 97 + K % 89 + M
    _check(w4, synth.gen_x(seed, M, K), seed, N, K, f"slots8 M={M} {N}x{K}")


@pytest.mark.parametrize("special", ["large", "tiny", "subnormal", "zeros"])
@pytest.mark.parametrize("M,N,K", [(8, 80000, 1536), (3, 80000, 1536), (8, 98304, 3072)])
def test_slots8_fp16_and_bf16_x(w4, special, M, N, K):
    # One x value outside fp16's exact range sends every CTA to the bf16 form;
    # exact zeros keep the fp16 one. K = 3072 at M = 8 stages bf16 regardless.
    seed = 5100 + M + N % 89
    x = synth.gen_x(seed, M, K).copy()
    r = M - 1
    if special == "large":
        x[r, 17] = 0x4980          # 2^20: beyond fp16's range
    elif special == "tiny":
        x[r, 300] = 0x3080         # 2^-30: below fp16's subnormal grid
    elif special == "subnormal":
        x[r, 5] = 0x0001           # a bf16 subnormal
    elif special == "zeros":
        x[:, 64:96] = 0x0000
    _check(w4, x, seed, N, K, f"slots8 x {special} M={M} {N}x{K}")


def test_slots8_zero_codes_exact(w4):
    # All codes 8: every product is an exact zero, in either unpack form.
    import torch
    for M, N, K in [(8, 80000, 1536), (4, 98304, 3072)]:
        x = synth.gen_x(5200, M, K)
        qw = to_dev_u32(np.full((N, K // 8), 0x88888888, dtype=np.uint32))
        sc = synth.gen_scales(5201, N, K)
        y = w4.w4a16_gemv(to_dev_bits16(x), qw, to_dev_bits16(sc))
        torch.cuda.synchronize()
        assert not torch.any(y).item(), (M, N, K)


def test_slots8_deterministic(w4):
    import torch
    for M, N, K in [(8, 80000, 1536), (5, 98304, 3072)]:
        seed = 5300 + M
        x = to_dev_bits16(synth.gen_x(seed, M, K))
        qd = synth.gen_qweight_torch(seed, N, K, "cuda")
        sd = to_dev_bits16(synth.gen_scales(seed, N, K))
        ys = [w4.w4a16_gemv(x, qd, sd) for _ in range(3)]
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32)), (M, N, K)


def _oracle_all_rows(x, qw, sc):
    """oracle.gemm over every row, in row ranges on the host's cores (the
    oracle's C loop runs without Python's lock)."""
    import concurrent.futures as cf
    import os
    N = qw.shape[0]
    parts = max(1, min(16, os.cpu_count() or 1))
    bounds = np.linspace(0, N, parts + 1).astype(np.int64)
    with cf.ThreadPoolExecutor(parts) as ex:
        res = list(ex.map(lambda i: oracle.gemm(x, qw, sc, rows=np.arange(bounds[i], bounds[i + 1])),
                          range(parts)))
    return np.concatenate([r[0] for r in res], axis=1), np.concatenate([r[1] for r in res], axis=1)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_slots8_vocab_argmax(w4, M):
    # The vocabulary projection 262144 x 1536 for M x-rows: logits on sampled
    # rows against the oracle and the greedy pick of every x-row exact (the
    # oracle's pick over all rows, with a gap beyond the bound).
    import torch
    N, K, seed = 262144, 1536, 5400 + M
    x = synth.gen_x(seed, M, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    y, a = y.cpu().numpy(), a.cpu().numpy()
    rows = np.unique(np.concatenate([[0, 1, N - 1], np.arange(13, N, 2053)]))
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(seed, N, K, rows), sc[rows])
    assert_w4_close(y[:, rows], yr, ar, what=f"slots8 vocab M={M}")
    qw = qd.cpu().numpy().view(np.uint32)
    yf, af = _oracle_all_rows(x, qw, sc)
    for m in range(M):
        idx, gap = oracle.argmax(yf[m])
        assert gap > 2 * (1e-4 * af[m, idx] + 1e-6), "ambiguous seed"
        assert int(a[m]) == idx, (m, int(a[m]), idx)
        assert int(a[m]) == int(np.argmax(y[m]))
