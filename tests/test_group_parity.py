"""Group sizes other than 32 (64, 128, 256, 512 codes per step) on every kernel,
against the fp64 oracle, through the C ABI.

Source: "fastgemma-gemma-4-E2B" model card, file table (FFN and LM-head weights
in int4 with group 256, the per-layer table with group 64) and its group-512
build; the format is otherwise the checkpoint paragraph's (codes 0..15, zero
point 8, one bf16 step per group along K).

Bars as for group 32: decode |y - y_ref| <= 1e-4 * sum|w x| + 1e-6; prefill
2e-3 * sum|w x|; gather and argmax bit-exact.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, bits16, to_dev_bits16, to_dev_u32
from _guard import guarded

pytestmark = pytest.mark.gpu

GROUPS = (64, 128, 256, 512)


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


def _problem(seed, M, N, K, group):
    return (synth.gen_x(seed, M, K), synth.gen_qweight(seed, N, K), synth.gen_scales(seed, N, K, group))


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("M,N,K", [(1, 2560, 1536), (2, 300, 2048), (1, 1536, 6144), (8, 2560, 1536),
                                   (5, 100, 1024), (1, 70, 512)])
def test_decode_groups(w4, group, M, N, K):
    import torch
    if K % group:
        pytest.skip("K not a multiple of the group")
    x, qw, sc = _problem(700 + M + N + group, M, N, K, group)
    y = w4.w4a16_gemv(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"decode g{group} M{M} N{N} K{K}")


@pytest.mark.parametrize("M", [1, 5])
def test_decode_group64_k_not_tile_multiple(w4, M):
    """K = 320: a multiple of the group (64) but not of the 128-code k-tile, the
    only group above 32 that reaches the guarded load paths (M <= 2 kernel and
    the 32-bit M <= 8 kernel)."""
    import torch
    N, K, group = 48, 320, 64
    x, qw, sc = _problem(760 + M, M, N, K, group)
    y = w4.w4a16_gemv(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"decode g64 K320 M{M}")


@pytest.mark.parametrize("M", [1, 2, 8])
def test_large_n_group256_argmax(w4, M):
    """The vocabulary-projection form (persistent kernel) with the LM head's group 256."""
    import torch
    N, K, group = 80000, 1536, 256
    x, qw, sc = _problem(780 + M, M, N, K, group)
    q = synth.gen_qweight_torch(780 + M, N, K, torch.device("cuda"))
    assert np.array_equal(q[:4].cpu().numpy().view(np.uint32), qw[:4])
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), q, to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, N, 997), [N - 1]]))
    yr, ar = oracle.gemm(x, qw[rows], sc[rows], group)
    assert_w4_close(y[:, rows], yr, ar, what=f"large-N g256 M{M}")
    yfull, afull = oracle.gemm(x, qw, sc, group)
    for m in range(M):
        idx, gap = oracle.argmax(yfull[m])
        assert gap > 2 * (1e-4 * afull[m, idx] + 1e-6), "ambiguous seed"
        assert int(a.cpu().numpy()[m]) == idx


@pytest.mark.parametrize("M,K,group", [(3, 8192, 64), (5, 8192, 128), (2, 32768, 32), (1, 8192, 256)])
def test_large_n_long_k(w4, M, K, group):
    """The persistent large-N forms where two CTAs' x staging no longer fits one
    SM's shared memory (M * K * 2 bytes each): the planner runs one CTA per SM.
    M = 3 and 5 take the M <= 8 form with one shared step per pair of groups
    (group 64) and a shifted step index (group 128); M = 2 at K = 32768 the M <= 2
    form. Sampled rows against the oracle; the pick equals the lowest index of
    the largest logit the kernel wrote."""
    import torch
    N = 78000
    x = synth.gen_x(800 + M, M, K)
    sc = synth.gen_scales(801 + M, N, K, group)
    q = synth.gen_qweight_torch(801 + M, N, K, torch.device("cuda"))
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), q, to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    y, a = y.cpu().numpy(), a.cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, N, 1013), [N - 17, N - 1]]))
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(801 + M, N, K, rows), sc[rows], group)
    assert_w4_close(y[:, rows], yr, ar, what=f"large N M{M} K{K} g{group}")
    for m in range(M):
        assert a[m] == int(np.argmax(y[m])), (m, a[m])


@pytest.mark.parametrize("group", (64, 256, 512))
def test_noalloc_groups(w4, group):
    import torch
    M, N, K = 1, 4096, 2048
    x, qw, sc = _problem(790 + group, M, N, K, group)
    y, a = w4.w4a16_gemv_argmax_noalloc(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"noalloc g{group}")
    assert int(a.cpu().numpy()[0]) == oracle.argmax(yr[0])[0]


@pytest.mark.parametrize("group", GROUPS)
def test_prefill_groups(w4, group):
    import torch
    M, N, K = 300, 384, 2048
    x, qw, sc = _problem(800 + group, M, N, K, group)
    y = w4.w4a16_gemm(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y.cpu().numpy(), yr, ar, rel=2e-3, abs_=0.0, what=f"prefill g{group}")
    assert w4.device_error() == 0


@pytest.mark.parametrize("group", GROUPS)
def test_gather_groups_bit_exact(w4, group):
    import torch
    N, K = 1000, 8960 if 8960 % group == 0 else 8192
    qt = synth.gen_qweight(810 + group, N, K)
    sc = synth.gen_scales(810 + group, N, K, group)
    ids = synth.gen_ids(811 + group, 8, N)
    ids_d = torch.from_numpy(ids.astype(np.int32)).cuda()
    out = w4.w4_embed_gather(ids_d, to_dev_u32(qt), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    ref, flag = oracle.embed_gather(ids, qt, sc, group)
    assert flag == 0
    np.testing.assert_array_equal(bits16(out), ref)


def test_rejected_group_sizes(w4):
    """Through the C entry point (validation runs before any buffer is read)."""
    import ctypes
    import torch
    x, qw, sc = _problem(820, 1, 64, 1024, 32)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    y = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    for group in (16, 48, 1024):
        rc = w4._lib.w4a16_gemv(P(y.data_ptr()), P(xd.data_ptr()), P(qd.data_ptr()), P(sd.data_ptr()),
                                1, 64, 1024, group, None)
        assert rc == 2, (group, rc)
