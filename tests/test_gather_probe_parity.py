"""GPU 4-bit row gather and memory read probe against the oracle (bit-exact)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from _util import bits16, to_dev_bits16, to_dev_u32
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


def _gather(w4, ids, qt, sc, qt_dev=None, status=None):
    import torch
    ids_d = torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()
    q = qt_dev if qt_dev is not None else to_dev_u32(qt)
    out = w4.w4_embed_gather(ids_d, q, to_dev_bits16(sc), status=status)
    torch.cuda.synchronize()
    return bits16(out)


def test_gather_hand_worked(w4):
    g = json.load(open(os.path.join(GOLDEN, "hand_2x64.json")))
    rows = [g["rows"]["r0"], g["rows"]["r1"]]
    qt = np.array([[int(w, 16) for w in r["words_hex"]] for r in rows], dtype=np.uint32)
    sc = np.array([[int(s, 16) for s in r["steps_bf16_hex"]] for r in rows], dtype=np.uint16)
    out = _gather(w4, [1, 0, 1], qt, sc)
    vals = synth.bf16_bits_to_f32(out[0]).astype(np.float64)
    assert vals[:8].tolist() == g["gather_r1"]["first8_values"]
    assert vals[32:36].tolist() == g["gather_r1"]["k32_to_35_values"]
    ref, _ = oracle.embed_gather(np.array([1, 0, 1]), qt, sc)
    assert np.array_equal(out, ref)


def test_gather_rounding_hand_worked(w4):
    g = json.load(open(os.path.join(GOLDEN, "bf16_rne.json")))
    step = int(g["step_bf16_hex"], 16)
    codes = [c["code"] for c in g["cases"]]
    qt = np.zeros((len(codes), 4), dtype=np.uint32)
    for i, c in enumerate(codes):
        w = 0
        for j in range(8):
            w |= c << (4 * j)
        qt[i, :] = w
    sc = np.full((len(codes), 1), step, dtype=np.uint16)
    out = _gather(w4, list(range(len(codes))), qt, sc)
    for i, c in enumerate(g["cases"]):
        assert np.all(out[i] == int(c["bf16_hex"], 16)), c


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (5, 33, 96), (64, 1000, 8960), (3, 7, 1536)])
def test_gather_random_bit_exact(w4, M, N, K):
    qt = synth.gen_qweight(80 + K, N, K)
    sc = synth.gen_scales(80 + K, N, K)
    ids = synth.gen_ids(81 + K, M, N)
    out = _gather(w4, ids, qt, sc)
    ref, flag = oracle.embed_gather(ids, qt, sc)
    assert flag == 0 and np.array_equal(out, ref)


def test_gather_out_of_range_ids(w4):
    import torch
    qt = synth.gen_qweight(90, 10, 64)
    sc = synth.gen_scales(90, 10, 64)
    ids = [3, 10, -2, 9]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gather(w4, ids, qt, sc, status=status)
    ref, flag = oracle.embed_gather(np.array(ids), qt, sc)
    assert flag == 1 and int(status.item()) == 1
    assert np.array_equal(out, ref)
    status.zero_()
    _gather(w4, [0, 9], qt, sc, status=status)
    assert int(status.item()) == 0


def test_gather_per_layer_table_8_ids(w4):
    # 262144 x 8960 table (35 x 256 values per token), group 32, 8 random ids.
    import torch
    N, K, seed = 262144, 8960, 2001
    qd = synth.gen_qweight_torch(seed, N, K, "cuda")
    sc = synth.gen_scales(seed, N, K)
    ids = synth.gen_ids(2002, 8, N)
    out = _gather(w4, ids, None, sc, qt_dev=qd)
    del qd
    torch.cuda.empty_cache()
    qrows = synth.gen_qweight_rows(seed, N, K, ids)
    ref, flag = oracle.embed_gather(np.arange(8), qrows, sc[ids])
    assert flag == 0 and np.array_equal(out, ref)


@pytest.mark.parametrize("nwords", [4, 1028, 3 * (1 << 20) + 4, 1 << 26])
def test_read_probe_sum(w4, nwords):
    import torch
    w = synth.gen_words(7, nwords)
    s = w4.hbm_read_probe(to_dev_u32(w))
    torch.cuda.synchronize()
    got = int(s.item()) & 0xFFFFFFFFFFFFFFFF
    assert got == oracle.sum_words(w)


def test_read_probe_closed_form(w4):
    import torch
    n = 1 << 22
    buf = torch.arange(n, dtype=torch.int32, device="cuda")
    s = w4.hbm_read_probe(buf)
    torch.cuda.synchronize()
    assert int(s.item()) == n * (n - 1) // 2


def test_gather_word_aligned_table_takes_the_word_path(w4):
    """A table only 4-byte aligned (allowed by the header) is gathered one word
    per thread; a 16-byte-aligned one a group per thread. Both bit-exact."""
    import torch
    N, K = 300, 2048
    qt = synth.gen_qweight(870, N, K)
    sc = synth.gen_scales(870, N, K)
    ids = synth.gen_ids(871, 64, N)
    ref, _ = oracle.embed_gather(ids, qt, sc)
    flat = torch.empty(N * (K // 8) + 1, dtype=torch.int32, device="cuda")
    flat[1:] = torch.from_numpy(qt.view(np.int32).ravel()).cuda()
    q_word = flat[1:].view(N, K // 8)
    assert q_word.data_ptr() % 16 != 0
    ids_d = torch.from_numpy(ids.astype(np.int32)).cuda()
    for q in (q_word, to_dev_u32(qt)):
        out = w4.w4_embed_gather(ids_d, q, to_dev_bits16(sc))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits16(out), ref)
