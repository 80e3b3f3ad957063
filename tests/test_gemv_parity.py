"""GPU decode GEMV/GEMM (M <= 8) against the fp64 oracle, through the C ABI.

Bar: |y - y_ref| <= 1e-4 * sum|w x| + 1e-6 elementwise; exact where the exact
result is representable (hand examples, all-8 codes, power-of-two scaling);
argmax index identical to the oracle's.
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


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


def _run(w4, x, qw, sc, argmax=False):
    import torch
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    if argmax:
        y, a = w4.w4a16_gemv_argmax(xd, qd, sd)
        torch.cuda.synchronize()
        return y.cpu().numpy(), a.cpu().numpy()
    y = w4.w4a16_gemm(xd, qd, sd)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_config0_full(w4):
    # One W4A16 GEMV, M=1, N=K=2048, seed 0.
    x, qw, sc = synth.gen_w4_problem(0, 1, 2048, 2048)
    y = _run(w4, x, qw, sc)
    yr, ar = oracle.gemm(x, qw, sc)
    worst = assert_w4_close(y, yr, ar, what="config0")
    assert worst < 1e-5


def test_hand_worked_examples_exact(w4):
    g = json.load(open(os.path.join(GOLDEN, "hand_2x64.json")))
    rows = [g["rows"]["r0"], g["rows"]["r1"]]
    qw = np.array([[int(w, 16) for w in r["words_hex"]] for r in rows], dtype=np.uint32)
    sc = np.array([[int(s, 16) for s in r["steps_bf16_hex"]] for r in rows], dtype=np.uint16)
    k = np.arange(64)
    xs = {"ones": np.ones(64), "ramp": k.astype(float),
          "alt": np.where(k % 2 == 0, 1.0, -1.0) * (1 + (k % 4) / 4)}
    for case in g["cases"]:
        x = synth.f64_to_bf16_bits(xs[case["x"]])[None, :]
        y = _run(w4, x, qw, sc)
        assert y[0].tolist() == case["y"], case["x"]
    # M = 3 and M = 8 kernels on the same rows
    x3 = np.stack([synth.f64_to_bf16_bits(xs[c]) for c in ("ones", "ramp", "alt")])
    y3 = _run(w4, x3, qw, sc)
    assert y3.tolist() == [c["y"] for c in g["cases"]]
    x8 = np.concatenate([x3, x3, x3[:2]])
    y8 = _run(w4, x8, qw, sc)
    assert y8.tolist() == [c["y"] for c in g["cases"]] * 2 + [g["cases"][0]["y"], g["cases"][1]["y"]]


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 32), (1, 17, 96), (1, 300, 160), (1, 33, 4192), (1, 64, 12288),
    (2, 45, 2080), (2, 1, 64), (2, 1000, 416),
    # K % 256 == 0 with M <= 2 runs the bulk-copy streaming kernel
    (1, 1, 256), (1, 17, 256), (2, 300, 512), (1, 33, 4352), (2, 777, 1536), (1, 70, 768),
    (2, 96, 2048), (1, 4097, 6144),
    (3, 19, 64), (4, 1, 96), (5, 40, 224), (7, 300, 1056), (8, 16, 32), (8, 129, 1536),
])
def test_ragged_shapes(w4, M, N, K):
    x, qw, sc = synth.gen_w4_problem(100 + M * 7 + N, M, N, K)
    y = _run(w4, x, qw, sc)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what=f"M{M} N{N} K{K}")


@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_all_codes_eight_give_exact_zero(w4, M):
    N, K = 70, 1536
    qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    sc = synth.gen_scales(5, N, K)
    x = synth.gen_x(5, M, K)
    y = _run(w4, x, qw, sc)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_power_of_two_steps_scale_bit_exactly(w4, M):
    x, qw, sc = synth.gen_w4_problem(41, M, 96, 2048)
    y = _run(w4, x, qw, sc)
    sc8 = (sc.astype(np.uint32) + (3 << 7)).astype(np.uint16)  # steps x 8
    y8 = _run(w4, x, qw, sc8)
    assert np.array_equal(y8, (8.0 * y).astype(np.float32))
    yn = _run(w4, x ^ np.uint16(0x8000), qw, sc)
    assert np.array_equal(yn, -y)


def test_run_to_run_bitwise_identical(w4):
    x, qw, sc = synth.gen_w4_problem(42, 1, 4096, 6144)
    a = _run(w4, x, qw, sc)
    b = _run(w4, x, qw, sc)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# The decode weight sweep's matrix shapes (N x K), unfused and fused.
SWEEP_SHAPES = [(2048, 1536), (256, 1536), (1536, 2048), (6144, 1536), (1536, 6144),
                (12288, 1536), (1536, 12288), (2560, 1536), (24576, 1536)]


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("N,K", SWEEP_SHAPES)
def test_sweep_shapes_sampled_rows(w4, M, N, K):
    import torch
    seed = 500 + N + K
    x = synth.gen_x(seed, M, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y = w4.w4a16_gemm(to_dev_bits16(x), qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 62)]))
    qrows = synth.gen_qweight_rows(seed, N, K, rows)
    yr, ar = oracle.gemm(x, qrows, sc[rows])
    assert_w4_close(y[:, rows], yr, ar, what=f"sweep {N}x{K} M{M}")


def test_device_qweight_generator_matches_host():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    a = synth.gen_qweight(9, 300, 1536)
    b = synth.gen_qweight_torch(9, 300, 1536, "cuda").cpu().numpy().view(np.uint32)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_argmax_small(w4, M):
    x, qw, sc = synth.gen_w4_problem(60 + M, M, 777, 1536)
    y, a = _run(w4, x, qw, sc, argmax=True)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what="argmax logits")
    for m in range(M):
        idx, gap = oracle.argmax(yr[m])
        tol = 1e-4 * ar[m, idx] + 1e-6
        assert gap > 2 * tol, "ambiguous seed"
        assert a[m] == idx
        assert a[m] == int(np.argmax(y[m]))


def test_argmax_ties_pick_lowest_index(w4):
    K, N = 1536, 200
    x, qw, sc = synth.gen_w4_problem(70, 1, N, K)
    yr, _ = oracle.gemm(x, qw, sc)
    top = int(np.argmax(yr[0]))
    for dup in (0, 17, top // 2):
        q2, s2 = qw.copy(), sc.copy()
        if dup == top:
            continue
        q2[dup], s2[dup] = qw[top], sc[top]
        y, a = _run(w4, x, q2, s2, argmax=True)
        first = int(np.flatnonzero(y[0] == y[0].max())[0])
        assert a[0] == first
        assert a[0] == min(dup, top)


def test_vocab_projection_with_argmax(w4):
    # N=262144 rows x K=1536, M=1, seed 1000: fp32 logits plus the fused greedy pick.
    import torch
    N, K, seed = 262144, 1536, 1000
    x = synth.gen_x(seed, 1, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    y, a = y.cpu().numpy(), a.cpu().numpy()
    qw = qd.cpu().numpy().view(np.uint32)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what="vocab")
    idx, gap = oracle.argmax(yr[0])
    assert gap > 2 * (1e-4 * ar[0, idx] + 1e-6), "ambiguous seed"
    assert int(a[0]) == idx
    assert int(a[0]) == int(np.argmax(y[0]))


@pytest.mark.parametrize("special", ["none", "large", "tiny", "subnormal", "zeros"])
@pytest.mark.parametrize("N,K,group", [(262144, 1536, 32), (131072, 3072, 256), (80000, 1536, 32)])
def test_fp16_and_bf16_unpack_forms(w4, special, N, K, group):
    """The kernels run an fp16 unpack when every x value is exact in fp16 and
    the bf16 one otherwise. x values outside fp16's exact range (2^20, 2^-30, a
    bf16 subnormal) force the bf16 form; x with exact zeros keeps the fp16 one.
    Both must meet the bound on sampled rows, and the pick must be the lowest
    index of the largest logit written."""
    import torch
    seed = 1300 + K + group
    x = synth.gen_x(seed, 1, K).copy()
    if special == "large":
        x[0, 17] = 0x4980          # 2^20: beyond fp16's range
    elif special == "tiny":
        x[0, 300] = 0x3080         # 2^-30: below fp16's subnormal grid
    elif special == "subnormal":
        x[0, 5] = 0x0001           # a bf16 subnormal
    elif special == "zeros":
        x[0, 64:96] = 0x0000
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K, group)
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), qd, to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    y, a = y.cpu().numpy(), a.cpu().numpy()
    rows = np.unique(np.concatenate([[0, N - 1], np.arange(7, N, 4099)]))
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(seed, N, K, rows), sc[rows], group)
    assert_w4_close(y[:, rows], yr, ar, what=f"x {special} {N}x{K} g{group}")
    assert int(a[0]) == int(np.argmax(y[0]))


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_large_n_sampled_rows_and_argmax(w4, M):
    # N = 80000 (5000 row blocks: the persistent large-N forms on a 152-SM GPU,
    # M <= 2 and M <= 8), K = 1536; logits on sampled rows plus the exact greedy
    # pick per x-row.
    import torch
    N, K, seed = 80000, 1536, 1100 + M
    x = synth.gen_x(seed, M, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    y, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), qd, to_dev_bits16(sc))
    y2 = w4.w4a16_gemv(to_dev_bits16(x), qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    y, a, y2 = y.cpu().numpy(), a.cpu().numpy(), y2.cpu().numpy()
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 15, 16, N - 1], rng.integers(0, N, 60)]))
    qrows = synth.gen_qweight_rows(seed, N, K, rows)
    yr, ar = oracle.gemm(x, qrows, sc[rows])
    assert_w4_close(y[:, rows], yr, ar, what=f"large N M{M}")
    for m in range(M):
        top = int(np.argmax(y[m]))
        assert int(a[m]) == int(np.flatnonzero(y[m] == y[m].max())[0]) == top
        # The picked row agrees with the oracle's value there.
        yt, at = oracle.gemm(x[m:m + 1], synth.gen_qweight_rows(seed, N, K, np.array([top])), sc[[top]])
        assert abs(float(y[m, top]) - yt[0, 0]) <= 1e-4 * at[0, 0] + 1e-6


@pytest.mark.parametrize("M", [1, 8])
def test_streaming_and_register_kernels_agree_with_oracle(w4, M):
    # Steps that are 4- but not 8- or 16-byte aligned take the kernels' narrow-load
    # paths; aligned ones the wide-load paths. Both agree with the oracle.
    import torch
    x, qw, sc = synth.gen_w4_problem(77, M, 500, 1536)
    yr, ar = oracle.gemm(x, qw, sc)
    xd, qd = to_dev_bits16(x), to_dev_u32(qw)
    flat = torch.zeros(sc.size + 8, dtype=torch.int16, device="cuda")
    flat[2:2 + sc.size] = torch.from_numpy(sc.view(np.int16).ravel()).cuda()
    sc_mis = flat[2:2 + sc.size].view(sc.shape)
    sc_al = to_dev_bits16(sc)
    assert sc_mis.data_ptr() % 16 != 0 and sc_al.data_ptr() % 16 == 0
    for s_dev in (sc_al, sc_mis):
        y = w4.w4a16_gemv(xd, qd, s_dev)
        torch.cuda.synchronize()
        assert_w4_close(y.cpu().numpy(), yr, ar, what="path")


def test_no_device_error_reported(w4):
    assert w4.device_error() == 0


def test_large_n_m8_steps_only_4_byte_aligned(w4):
    """The M <= 8 large-N form with a step table 4-byte but not 8-byte aligned
    (allowed by the header): the step loads fall back to 16-bit ones; same bits
    as the 8-byte-aligned call."""
    import torch
    M, N, K, seed = 8, 80000, 1536, 1190
    x = synth.gen_x(seed, M, K)
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    flat = torch.empty(N * (K // 32) + 2, dtype=torch.int16, device="cuda")
    flat[2:] = torch.from_numpy(sc.view(np.int16).ravel()).cuda()
    sc4 = flat[2:].view(N, K // 32)
    assert sc4.data_ptr() % 8 == 4
    xd = to_dev_bits16(x)
    y4, a4 = w4.w4a16_gemv_argmax(xd, qd, sc4)
    y8, a8 = w4.w4a16_gemv_argmax(xd, qd, to_dev_bits16(sc))
    torch.cuda.synchronize()
    assert torch.equal(y4, y8) and torch.equal(a4, a8)
    rows = np.array([0, 1, 40000, N - 1])
    yr, ar = oracle.gemm(x, synth.gen_qweight_rows(seed, N, K, rows), sc[rows])
    assert_w4_close(y4.cpu().numpy()[:, rows], yr, ar, what="large N M8, 4-byte-aligned steps")


@pytest.mark.parametrize("M", [3, 5, 8])
@pytest.mark.parametrize("N,K", [(1536, 12288), (1536, 6144), (64, 4096), (608, 8192), (1530, 6144),
                                 (60, 4096)])
def test_m8_cluster_k_quarters(w4, M, N, K):
    """The M <= 8 form whose 1536-row long-K calls run as clusters of 4 CTAs
    (each CTA a K quarter of 4 row blocks, the quarters added by the owning
    CTA in rank order): every row against the oracle, all-8 codes exactly zero,
    and run to run bitwise identical. 1530 and 60 rows end in a ragged row
    block inside a cluster; 608 rows (38 row blocks) take the one-CTA form."""
    import torch
    x, qw, sc = synth.gen_w4_problem(5600 + M + N % 97 + K % 89, M, N, K)
    y = _run(w4, x, qw, sc)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what=f"cluster M{M} N{N} K{K}")
    y2 = _run(w4, x, qw, sc)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))
    z = _run(w4, x, np.full_like(qw, 0x88888888), sc)
    assert not np.any(z)


_CAPTURE_FIRST = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import synth, bit_weight_only_w4a16_gb300 as w4
from _util import to_dev_bits16, to_dev_u32
w4.init()
x, qw, sc = synth.gen_w4_problem(5700, 8, 1536, 12288)
xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
y = torch.empty((8, 1536), dtype=torch.float32, device="cuda")
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):  # the first M = 8 call of the process
    w4.w4a16_gemm(xd, qd, sd, out=y, stream=s)
g.replay(); torch.cuda.synchronize()
ref = w4.w4a16_gemm(xd, qd, sd); torch.cuda.synchronize()
assert torch.equal(y, ref), "replayed graph differs from the eager call"
np.save(sys.argv[1], y.cpu().numpy())
"""


def test_m8_cluster_form_captured_as_first_call(w4, tmp_path):
    """A process whose first M = 8 call (a cluster-form shape) is made under
    stream capture: the per-device set-up has done the one-time queries, so
    the capture succeeds, and the replayed graph gives the eager call's bits
    and the oracle's values."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = tmp_path / "y.npy"
    code = _CAPTURE_FIRST.format(root=root, tests=os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code, str(out)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    x, qw, sc = synth.gen_w4_problem(5700, 8, 1536, 12288)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(np.load(out), yr, ar, what="captured first M=8 call")
