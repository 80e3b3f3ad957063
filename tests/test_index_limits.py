"""The largest weight table the entry points accept: N * K/8 just below 2^31
words (K = 8192, N = 2,097,136 rows: 8.6 GB of codes, 1.07 GB of steps). Every
kernel indexes rows with 64-bit offsets; this runs them at the limit and checks
sampled rows (first, middle, last and random) against the oracle, the greedy
pick for validity (the lowest index of the maximum of the device's own
outputs, which no oracle can form for 2 M rows in a test), and the gather of the
last rows bit-exactly.

Steps follow a row- and group-dependent pattern generated identically on the
device and for the sampled rows on the host (bf16 bits 0x3C00 + (37 r + 11 g)
mod 256: positive, 2^-7 .. 2^-5), so a step read from the wrong row shows.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, bits16, to_dev_bits16
from _guard import guarded

pytestmark = pytest.mark.gpu

K = 8192
N = ((2 ** 31 - 1) // (K // 8)) // 16 * 16


def _steps_host(rows):
    g = np.arange(K // 32, dtype=np.int64)[None, :]
    r = np.asarray(rows, dtype=np.int64)[:, None]
    return (0x3C00 + (37 * r + 11 * g) % 256).astype(np.uint16)


@pytest.fixture(scope="module")
def table():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    dev = torch.device("cuda")
    assert N * (K // 8) < 2 ** 31 and (N + 16) * (K // 8) >= 2 ** 31
    q = synth.gen_qweight_torch(1234, N, K, dev)
    sc = torch.empty((N, K // 32), dtype=torch.int16, device=dev)
    g = torch.arange(K // 32, device=dev, dtype=torch.int64)[None, :]
    for r0 in range(0, N, 1 << 18):
        r = torch.arange(r0, min(N, r0 + (1 << 18)), device=dev, dtype=torch.int64)[:, None]
        sc[r0:r0 + r.shape[0]] = (0x3C00 + (37 * r + 11 * g) % 256).to(torch.int16)
    torch.cuda.synchronize()
    rng = np.random.default_rng(55)
    rows = np.unique(np.concatenate([[0, 1, N // 2, N - 17, N - 16, N - 2, N - 1], rng.choice(N, 41, replace=False)]))
    return guarded(w4), q, sc, rows


@pytest.mark.parametrize("M", [1, 8])
def test_decode_at_the_index_limit(table, M):
    import torch
    w4, q, sc, rows = table
    x = synth.gen_x(1235 + M, M, K)
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), q, sc)
    torch.cuda.synchronize()
    assert w4.device_error() == 0
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(1234, N, K, rows), _steps_host(rows))
    assert_w4_close(y[:, rows].cpu().numpy(), yr, ar, what=f"index limit M={M}")
    for m in range(M):
        idx = int(a[m].item())
        row = y[m]
        top = row.max()
        assert row[idx] == top, (m, idx)
        assert not bool((row[:idx] == top).any()), "not the lowest index of the maximum"


def test_gather_at_the_index_limit(table):
    import torch
    w4, q, sc, rows = table
    ids = np.array([N - 1, 0, N // 2, N - 16], dtype=np.int32)
    out = w4.w4_embed_gather(torch.from_numpy(ids).cuda(), q, sc)
    torch.cuda.synchronize()
    ref, flag = oracle.embed_gather(np.arange(len(ids), dtype=np.int32), synth.gen_qweight_rows(1234, N, K, ids),
                                    _steps_host(ids))
    assert flag == 0
    np.testing.assert_array_equal(bits16(out), ref)
