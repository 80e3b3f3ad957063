"""The M = 1 decode form with K split over the warps of a CTA (the few-tiles-per-
warp form chosen for the small decode projections), against the fp64 oracle
through the C ABI.

The shapes cover the planner's choices: 8, 12 and 16 warps, one or two CTAs on
an SM, one or several 16-row blocks per CTA with a shorter last CTA, sub-slices
of equal and of unequal length, and group sizes 32 to 512; the decode sweep's
longer shapes (served by the shared-memory slot form) are checked here too,
with the slot form's largest CTA (16 row blocks x 2 slices = its 32 slots),
the same with a shorter last CTA, and the first shape past it (17 row blocks a
CTA: the register-preload form).
Bar: |y - y_ref| <= 1e-4 * sum|w x| + 1e-6 elementwise, and run to run bitwise
identical results (fixed-order sums, no atomics).
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


def _gemv(w4, x, qw, sc, group):
    import torch
    y = w4.w4a16_gemv(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc), group=group)
    torch.cuda.synchronize()
    return y.cpu().numpy()


# (N, K): the decode sweep's fused shapes, then shapes that reach the other
# plans: two row blocks per CTA (6160 x 768), unequal sub-slices (784 x 1152,
# 48 x 384, 16 x 1152), one tile per warp, 12 and 16 warps.
SHAPES = [(2560, 1536), (1536, 2048), (12288, 1536), (1536, 6144), (24576, 1536), (1536, 12288),
          (2048, 2048), (256, 1536), (16, 128), (4096, 1536), (48, 384), (1536, 128),
          (2576, 1536), (1552, 6144), (3088, 3072), (784, 1024), (400, 6144), (32768, 2048),
          (6160, 768), (1200, 8192), (784, 1152), (16, 1152), (38912, 1536), (38896, 1536),
          (38928, 1536)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_m1_shapes_group32(w4, N, K):
    x, qw, sc = synth.gen_w4_problem(4000 + N % 97 + K % 89, 1, N, K)
    y = _gemv(w4, x, qw, sc, 32)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what=f"m1 {N}x{K}")


@pytest.mark.parametrize("group", [64, 128, 256, 512])
@pytest.mark.parametrize("N,K", [(2560, 1536), (1536, 2048), (1552, 6144), (784, 1152), (1536, 12288)])
def test_m1_shapes_groups(w4, N, K, group):
    if K % group:
        pytest.skip("K not a multiple of the group")
    x = synth.gen_x(4100 + group, 1, K)
    qw = synth.gen_qweight(4101 + group, N, K)
    sc = synth.gen_scales(4102 + group, N, K, group)
    y = _gemv(w4, x, qw, sc, group)
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y, yr, ar, what=f"m1 {N}x{K} g{group}")


def test_m1_zero_codes_exact(w4):
    # All codes 8: every product is an exact zero, whatever the split.
    for N, K in [(1536, 2048), (2560, 1536), (1536, 6144)]:
        x = synth.gen_x(4200, 1, K)
        qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
        sc = synth.gen_scales(4201, N, K)
        y = _gemv(w4, x, qw, sc, 32)
        assert not np.any(y), (N, K)


def test_m1_deterministic(w4):
    import torch
    for N, K in [(1536, 2048), (1536, 6144), (2560, 1536)]:
        x, qw, sc = synth.gen_w4_problem(4300, 1, N, K)
        xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
        ys = [w4.w4a16_gemv(xd, qd, sd) for _ in range(3)]
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int32), ys[0].view(torch.int32)), (N, K)


@pytest.mark.parametrize("special", ["none", "large", "tiny", "subnormal", "zeros"])
@pytest.mark.parametrize("N,K", [(2560, 1536), (24576, 1536), (1536, 6144), (1536, 12288)])
def test_m1_special_x_values(w4, special, N, K):
    """The sweep's long M = 1 shapes with x values at the edges of bf16 (2^20,
    2^-30, a bf16 subnormal) and with runs of exact zeros: the bound against
    the oracle holds for each."""
    x, qw, sc = synth.gen_w4_problem(4400 + N % 89 + K % 83, 1, N, K)
    x = x.copy()
    if special == "large":
        x[0, 17] = 0x4980          # 2^20: beyond fp16's range
    elif special == "tiny":
        x[0, 300] = 0x3080         # 2^-30: below fp16's subnormal grid
    elif special == "subnormal":
        x[0, 5] = 0x0001           # a bf16 subnormal
    elif special == "zeros":
        x[0, 64:96] = 0x0000
    y = _gemv(w4, x, qw, sc, 32)
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y, yr, ar, what=f"m1 {N}x{K} x {special}")
