"""Pins of the decode-step plumbing oracle (no GPU).

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the cache paragraph
(full layers: one slot per position; sliding layers: a ring of slots recording
each slot's position), the CUDA-graph paragraph (every position kept on the
GPU), the emb4 paragraph (embedding and LM head share one 4-bit table) and the
tool-calling paragraph (a forced token skips the LM-head read).

Each pin fails on a plausible mistake: a ring slot off by one or not wrapped, a
slot table not updated (hand-written final state; ring attention equal to the
full-cache attention over the same window), a history index or position step
off by one, a row looked up from the wrong token, a forced token ignored, or a
greedy pick taken from the wrong row (hand-computed tables).
"""
import numpy as np

import oracle
import synth


def _val(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_ring_after_ten_appends_holds_the_last_four_positions():
    T, D = 4, 8
    kc = np.zeros((T, D), np.uint16)
    vc = np.zeros((T, D), np.uint16)
    kp = np.full(T, -1, np.int32)
    for p in range(10):
        row = np.full(D, 0x3F80 + p, np.uint16)  # a distinct bf16 pattern per position
        kc, vc, kp, st = oracle.kv_append(kc, vc, kp, row, row ^ 0x8000, p)
        assert st == 0
    # Positions 8, 9 wrote slots 0, 1 last; 6, 7 slots 2, 3.
    np.testing.assert_array_equal(kp, [8, 9, 6, 7])
    np.testing.assert_array_equal(kc[:, 0], [0x3F88, 0x3F89, 0x3F86, 0x3F87])
    np.testing.assert_array_equal(vc[:, 0], [0xBF88, 0xBF89, 0xBF86, 0xBF87])


def test_full_cache_append_and_out_of_range():
    T, D = 3, 8
    kc = np.zeros((T, D), np.uint16)
    vc = np.zeros((T, D), np.uint16)
    row = np.arange(D, dtype=np.uint16) + 1
    kc2, vc2, kp2, st = oracle.kv_append(kc, vc, None, row, row, 2)
    assert st == 0 and kp2 is None
    np.testing.assert_array_equal(kc2[2], row)
    assert not kc2[:2].any()
    for bad in (3, -1):
        kc3, vc3, _, st = oracle.kv_append(kc2, vc2, None, row * 2, row * 2, bad)
        assert st == 1
        np.testing.assert_array_equal(kc3, kc2)
    _, _, kp4, st = oracle.kv_append(kc, vc, np.full(T, -1, np.int32), row, row, -5)
    assert st == 1 and (kp4 == -1).all()


def test_ring_attention_equals_windowed_full_cache():
    """Appending positions 0..P-1 to a T-slot ring and attending with window T gives
    the attention over a full cache of the same positions restricted to the last
    T of them."""
    T, D, P, H = 16, 128, 41, 8
    q = synth.gen_attn_q(31, H, D)
    kall, vall = synth.gen_attn_kv(31, P, D)
    kc = np.zeros((T, D), np.uint16)
    vc = np.zeros((T, D), np.uint16)
    kp = np.full(T, -1, np.int32)
    for p in range(P):
        kc, vc, kp, st = oracle.kv_append(kc, vc, kp, kall[p], vall[p], p)
        assert st == 0
        ring, _ = oracle.attn_decode(q, kc, vc, kp, qpos=p, window=T, scale=0.1)
        full, _ = oracle.attn_decode(q, kall[:p + 1], vall[:p + 1], None, qpos=p, window=T, scale=0.1)
        np.testing.assert_allclose(ring, full, rtol=1e-12, atol=1e-15)


def _table():
    """V = 4 rows, K = 32 (one group of 32): row r holds code 8 + r - 1 everywhere
    (values (r - 1) * step), steps 0.5, 1, 2, 4."""
    V, K = 4, 32
    codes = np.array([7, 8, 9, 10], dtype=np.uint32)
    q = np.zeros((V, K // 8), np.uint32)
    for r in range(V):
        w = 0
        for j in range(8):
            w |= int(codes[r]) << (4 * j)
        q[r] = w
    sc = np.array([[0x3F00], [0x3F80], [0x4000], [0x4080]], np.uint16)  # 0.5, 1, 2, 4
    return q, sc


def test_prologue_hand_table():
    q, sc = _table()
    hist = np.full(6, -7, np.int32)
    x, hist2, pos, st = oracle.decode_prologue(3, 2, hist, q, sc, 32)
    assert pos == 3 and st == 0
    np.testing.assert_array_equal(hist2, [-7, -7, -7, 3, -7, -7])
    # row 3: (10 - 8) * 4 = 8.0 -> bf16 0x4100
    np.testing.assert_array_equal(x, np.full((1, 32), 0x4100, np.uint16))
    x, _, pos, st = oracle.decode_prologue(0, 0, hist, q, sc, 32)
    np.testing.assert_array_equal(x, np.full((1, 32), 0xBF00, np.uint16))  # (7 - 8) * 0.5 = -0.5
    assert pos == 1 and st == 0


def test_prologue_bad_token_and_full_history():
    q, sc = _table()
    hist = np.zeros(3, np.int32)
    x, hist2, pos, st = oracle.decode_prologue(4, 0, hist, q, sc, 32)
    assert st == 1 and pos == 1 and hist2[1] == 4
    assert not x.any()
    x, hist3, pos, st = oracle.decode_prologue(1, 2, hist, q, sc, 32)
    assert st == 2 and pos == 3
    np.testing.assert_array_equal(hist3, hist)
    np.testing.assert_array_equal(x, np.zeros((1, 32), np.uint16))  # row 1: code 8 -> 0
    _, _, pos, st = oracle.decode_prologue(2, 5, None, q, sc, 32)
    assert pos == 6 and st == 0


def test_lm_head_pick_forced_and_greedy():
    q, sc = _table()
    x = np.full((1, 32), 0x3F80, np.uint16)  # x = 1 everywhere
    # logits: row r = 32 * (r - 1) * step_r = -16, 0, 64, 256 -> greedy pick 3
    tok, y, a = oracle.lm_head_pick(x, q, sc, 32, -1)
    assert tok == 3
    np.testing.assert_array_equal(y[0], [-16.0, 0.0, 64.0, 256.0])
    tok, y, a = oracle.lm_head_pick(x, q, sc, 32, 1)
    assert tok == 1 and y is None and a is None
    xn = np.full((1, 32), 0xBF80, np.uint16)  # x = -1: logits 16, 0, -64, -256 -> pick 0
    assert oracle.lm_head_pick(xn, q, sc, 32, -1)[0] == 0
