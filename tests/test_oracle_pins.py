"""Pins of the CPU oracle against facts fixed outside it (no GPU needed).

Each pin is chosen so that a plausible mistake in the oracle fails at least one:
hand-worked examples with the packed words in hex (nibble order, zero point,
group boundary, step dtype), closed-form invariants, exact rational brute force
on tiny shapes, and hand-rounded bf16 values.
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _hand():
    g = _load("hand_2x64.json")
    rows = [g["rows"]["r0"], g["rows"]["r1"]]
    qw = np.array([[int(w, 16) for w in r["words_hex"]] for r in rows], dtype=np.uint32)
    sc = np.array([[int(s, 16) for s in r["steps_bf16_hex"]] for r in rows], dtype=np.uint16)
    return g, qw, sc


def _x_case(name, K=64):
    k = np.arange(K)
    if name == "ones":
        v = np.ones(K)
    elif name == "ramp":
        v = k.astype(np.float64)
    elif name == "alt":
        v = np.where(k % 2 == 0, 1.0, -1.0) * (1.0 + (k % 4) / 4.0)
    else:
        raise KeyError(name)
    return synth.f64_to_bf16_bits(v)[None, :]


# -- exact rational brute force, independent of the oracle's code path ---------

def _nibbles_by_hex(word):
    """Codes of one word via its hex text: the last hex digit is the first code."""
    return [int(c, 16) for c in reversed("%08x" % int(word))]


def _bf16_exact(bits):
    f = struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]
    return Fraction(f)


def _exact_gemm(x, qw, sc, group=32):
    M, K = x.shape
    N = qw.shape[0]
    y = [[Fraction(0)] * N for _ in range(M)]
    a = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        codes = []
        for w in qw[n]:
            codes.extend(_nibbles_by_hex(w))
        wn = [(codes[k] - 8) * _bf16_exact(sc[n][k // group]) for k in range(K)]
        for m in range(M):
            for k in range(K):
                t = _bf16_exact(x[m][k]) * wn[k]
                y[m][n] += t
                a[m][n] += abs(t)
    return y, a


def test_unpack_trick_is_exact_for_all_codes():
    # The w4gemv paragraph: OR a code into the bits of 2^23, subtract 2^23 + 8.
    for q in range(16):
        f = struct.unpack("<f", struct.pack("<I", 0x4B000000 | q))[0]
        assert np.float32(f) - np.float32(8388616.0) == q - 8
        # the same trick one bf16 at a time: 0x4300 | q is 128 + q.
        b = struct.unpack("<f", struct.pack("<I", (0x4300 | q) << 16))[0]
        assert b - 136.0 == q - 8


@pytest.mark.parametrize("case", ["ones", "ramp", "alt"])
def test_hand_worked_2x64(case):
    g, qw, sc = _hand()
    c = next(c for c in g["cases"] if c["x"] == case)
    y, a = oracle.gemm(_x_case(case), qw, sc)
    assert y[0].tolist() == c["y"]
    assert a[0].tolist() == c["absy"]


def test_hand_example_rejects_wrong_readings():
    """The r1/ramp pin separates the right reading from the plausible wrong ones."""
    g, qw, sc = _hand()
    want = next(c for c in g["cases"] if c["x"] == "ramp")["y"][1]
    wrong = g["wrong_readings_on_r1_ramp"]
    x = np.arange(64, dtype=np.float64)
    steps = [0.25, 2.0]

    def y_with(code_of):
        return sum(x[k] * code_of(k) * steps[k // 32] for k in range(64))

    words = qw[1]
    hi_first = lambda k: ((int(words[k // 8]) >> (4 * (7 - k % 8))) & 15) - 8
    signed = lambda k: (lambda c: c - 16 if c >= 8 else c)((int(words[k // 8]) >> (4 * (k % 8))) & 15)
    no_zero = lambda k: (int(words[k // 8]) >> (4 * (k % 8))) & 15
    got = {"high_nibble_first": y_with(hi_first),
           "signed_int4_twos_complement": y_with(signed),
           "zero_point_omitted": y_with(no_zero)}
    for name, v in got.items():
        assert v == wrong[name], name
        assert v != want


def test_gather_hand_worked():
    g, qw, sc = _hand()
    out, flag = oracle.embed_gather(np.array([1, 0], dtype=np.int32), qw, sc)
    vals = synth.bf16_bits_to_f32(out[0]).astype(np.float64)
    assert vals[:8].tolist() == g["gather_r1"]["first8_values"]
    assert vals[32:36].tolist() == g["gather_r1"]["k32_to_35_values"]
    assert flag == 0
    assert np.all(synth.bf16_bits_to_f32(out[1]) == np.float32(np.repeat([1.0, 0.5], 32)))


def test_gather_rounding_hand_worked():
    g = _load("bf16_rne.json")
    step = int(g["step_bf16_hex"], 16)
    K = 32
    for c in g["cases"]:
        word = 0
        for j in range(8):
            word |= c["code"] << (4 * j)
        qt = np.full((1, K // 8), word, dtype=np.uint32)
        sc = np.full((1, 1), step, dtype=np.uint16)
        out, _ = oracle.embed_gather(np.array([0], dtype=np.int32), qt, sc)
        assert np.all(out == int(c["bf16_hex"], 16)), c
        assert oracle.f32_to_bf16(c["exact"]) == int(c["bf16_hex"], 16)


def test_gather_out_of_range_ids_zero_fill_and_flag():
    qt = synth.gen_qweight(11, 4, 64)
    sc = synth.gen_scales(11, 4, 64)
    out, flag = oracle.embed_gather(np.array([2, 4, -1], dtype=np.int32), qt, sc)
    assert flag == 1
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    ref, flag0 = oracle.embed_gather(np.array([2], dtype=np.int32), qt, sc)
    assert flag0 == 0 and np.array_equal(out[0], ref[0])


def test_all_codes_eight_give_exact_zero():
    K, N = 256, 5
    qw = np.full((N, K // 8), 0x88888888, dtype=np.uint32)
    sc = synth.gen_scales(3, N, K)
    x = synth.gen_x(3, 2, K)
    y, a = oracle.gemm(x, qw, sc)
    assert np.all(y == 0.0) and np.all(a == 0.0)


def test_power_of_two_step_scaling_is_exact():
    x, qw, sc = synth.gen_w4_problem(21, 2, 6, 512)
    y, _ = oracle.gemm(x, qw, sc)
    sc4 = (sc.astype(np.uint32) + (2 << 7)).astype(np.uint16)  # exponent + 2: steps x 4
    y4, _ = oracle.gemm(x, qw, sc4)
    assert np.array_equal(y4, 4.0 * y)


def test_negated_x_negates_y_exactly():
    x, qw, sc = synth.gen_w4_problem(22, 1, 7, 256)
    y, _ = oracle.gemm(x, qw, sc)
    yn, _ = oracle.gemm(x ^ np.uint16(0x8000), qw, sc)
    assert np.array_equal(yn, -y)


def test_row_subset_matches_full():
    x, qw, sc = synth.gen_w4_problem(23, 3, 40, 192)
    y, a = oracle.gemm(x, qw, sc)
    rows = np.array([39, 0, 17, 17, 5])
    ys, as_ = oracle.gemm(x, qw, sc, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(as_, a[:, rows])


@pytest.mark.parametrize("seed,M,N,K", [(31, 1, 3, 32), (32, 2, 5, 96), (33, 3, 8, 128), (34, 1, 1, 64)])
def test_brute_force_exact_rationals(seed, M, N, K):
    x, qw, sc = synth.gen_w4_problem(seed, M, N, K)
    y, a = oracle.gemm(x, qw, sc)
    ye, ae = _exact_gemm(x, qw, sc)
    for m in range(M):
        for n in range(N):
            bound = K * 2.0 ** -52 * float(ae[m][n])
            assert abs(Fraction(y[m, n]) - ye[m][n]) <= Fraction(bound)
            assert abs(Fraction(a[m, n]) - ae[m][n]) <= Fraction(bound)


def test_dense_dequant_matches_exact_and_library_matmul():
    x, qw, sc = synth.gen_w4_problem(35, 3, 6, 160)
    w = oracle.dequant(qw, sc)
    for n in range(6):
        codes = []
        for word in qw[n]:
            codes.extend(_nibbles_by_hex(word))
        for k in range(160):
            assert Fraction(w[n, k]) == (codes[k] - 8) * _bf16_exact(sc[n][k // 32])
    y, a = oracle.gemm(x, qw, sc)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    np.testing.assert_allclose(y, xf @ w.T, rtol=0, atol=1e-12 * a.max())


def test_argmax_lowest_index_and_signed_zero():
    assert oracle.argmax(np.array([1.0, 3.0, 3.0, 2.0]))[0] == 1
    idx, gap = oracle.argmax(np.array([-0.0, 0.0, -1.0]))
    assert idx == 0 and gap == 0.0
    idx, gap = oracle.argmax(np.array([-5.0, -2.0, -3.5]))
    assert idx == 1 and gap == 1.5
    rng = np.random.default_rng(0)
    for _ in range(50):
        v = rng.integers(-3, 4, size=17).astype(np.float64)
        assert oracle.argmax(v)[0] == min(i for i in range(17) if v[i] == v.max())


def test_sum_words_closed_forms():
    n = 100000
    assert oracle.sum_words(np.arange(n, dtype=np.uint32)) == n * (n - 1) // 2
    assert oracle.sum_words(np.full(n, 0xFFFFFFFF, dtype=np.uint32)) == n * 0xFFFFFFFF
    w = synth.gen_words(1, 4097)
    assert oracle.sum_words(w) == int(w.astype(np.uint64).sum()) % (1 << 64)


def test_size_arithmetic_matches_the_pages():
    # Per-layer table: 262,144 tokens x 35 x 256 values; 4.375 GiB in 16-bit.
    assert 262144 * 35 * 256 * 2 == int(4.375 * 2 ** 30)
    # Embedding 262,144 x 1536 in 16-bit is 0.75 GiB.
    assert 262144 * 1536 * 2 == int(0.75 * 2 ** 30)
    # 1,222.8 MiB read in 9.12 ms is 140.6 GB/s.
    assert abs(1222.8 * 2 ** 20 / 9.12e-3 / 1e9 - 140.6) < 0.05


@pytest.mark.parametrize("group", [64, 128, 256, 512])
def test_group_equals_repeated_group32_steps(group):
    """A group-G step applies to G consecutive codes: the same problem written
    with group 32 and each step repeated G/32 times gives bit-identical y, |y|
    sums, dequantized weights and gathered rows (a wrong step index or row
    stride for G != 32 breaks this)."""
    M, N, K = 3, 5, 1024
    x = synth.gen_x(900 + group, M, K)
    qw = synth.gen_qweight(900 + group, N, K)
    scg = synth.gen_scales(900 + group, N, K, group)
    sc32 = np.repeat(scg, group // 32, axis=1)
    assert sc32.shape == (N, K // 32)
    y1, a1 = oracle.gemm(x, qw, scg, group)
    y2, a2 = oracle.gemm(x, qw, sc32, 32)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(oracle.dequant(qw, scg, group), oracle.dequant(qw, sc32, 32))
    ids = np.array([4, 0, 2], dtype=np.int32)
    g1, _ = oracle.embed_gather(ids, qw, scg, group)
    g2, _ = oracle.embed_gather(ids, qw, sc32, 32)
    np.testing.assert_array_equal(g1, g2)
