"""The shared input generator follows its published definitions."""
import numpy as np

import synth


def test_splitmix64_published_vector():
    # SplitMix64 from state 0: the first outputs of the reference generator.
    got = [int(v) for v in synth.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_slices_agree():
    s = synth.stream_state(9, 1)
    full = synth.splitmix64(s, 0, 1000)
    assert np.array_equal(full[300:700], synth.splitmix64(s, 300, 400))


def test_normals_moments_and_bf16_rounding():
    z = synth.normals(synth.stream_state(4, 2), 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    b = synth.f64_to_bf16_bits(np.array([1.0, 1.00390625, 1.01171875, -2.5, 0.0]))
    # 1 + 2^-8 is a tie between 1.0 and 1 + 2^-7: even wins (1.0).
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: even wins (1 + 2^-6).
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]


def test_distributions():
    sc = synth.bf16_bits_to_f32(synth.gen_scales(1, 64, 1024)).astype(np.float64)
    assert sc.min() >= 1e-4 * 0.99 and abs(sc.mean() - (0.02 * np.sqrt(2 / np.pi) + 1e-4)) < 1e-3
    q = synth.gen_qweight(1, 64, 1024)
    nib = np.stack([(q >> (4 * j)) & 15 for j in range(8)])
    counts = np.bincount(nib.ravel(), minlength=16)
    assert counts.min() > 0.9 * counts.mean()
    ids = synth.gen_ids(2002, 1000, 262144)
    assert ids.min() >= 0 and ids.max() < 262144
