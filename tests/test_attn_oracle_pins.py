"""Pins of the decode-attention oracle against facts fixed outside it (no GPU).

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the decode-attention
paragraph (one key/value head read once for eight query heads, a softmax over
the cached positions, then the values) and the cache paragraph (full layers: one
slot per position, one head of width 512, 2 KiB per token per layer; sliding
layers: a 512-slot ring that records each slot's position; 774 MiB for a
131,072-token context); "Step 4 - The Model in Rust" (the ring keeps a slot only
when its position is >= 0, not after the query and, with a window w, after the
query's position minus w).

Each pin fails on a plausible oracle mistake: a dropped max-subtraction or
normalisation (closed forms), a wrong mask boundary (ring rules), a transposed
operand or wrong scale (library softmax on a random case), weights applied to
the wrong slot (permutation, single slot).
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _bits(a):
    return synth.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def _val(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_single_kept_slot_returns_its_value():
    q = synth.gen_attn_q(11, 8, 64)
    k, v = synth.gen_attn_kv(11, 6, 64)
    kpos = np.array([-1, 9, 3, 7, 2, -1], dtype=np.int32)  # qpos 3, window 1: only position 3 kept
    out, absout = oracle.attn_decode(q, k, v, kpos, qpos=3, window=1, scale=0.3)
    np.testing.assert_array_equal(out, np.broadcast_to(_val(v[2]), out.shape))
    np.testing.assert_array_equal(absout, np.broadcast_to(np.abs(_val(v[2])), out.shape))


def test_zero_query_gives_mean_of_kept_values():
    q = np.zeros((8, 32), dtype=np.uint16)
    k, v = synth.gen_attn_kv(12, 40, 32)
    kpos = synth.ring_positions(57, 40)
    out, _ = oracle.attn_decode(q, k, v, kpos, qpos=57, window=25, scale=1.0)
    keep = (kpos >= 0) & (kpos <= 57) & (kpos > 57 - 25)
    ref = _val(v[keep]).mean(axis=0)
    np.testing.assert_allclose(out, np.broadcast_to(ref, out.shape), rtol=1e-14, atol=1e-15)


def test_two_slot_closed_form():
    # scores (0, s) for q = e0 and keys 0 and e0: weights 1/(1+e^s), e^s/(1+e^s).
    D = 4
    q = _bits([[1.0, 0.0, 0.0, 0.0]])
    k = _bits([[0.0, 0.0, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0]])
    v = _bits([[2.0, 0.0, -1.0, 0.5], [-4.0, 1.0, 3.0, 0.5]])
    for scale in (1.0, 0.5, 2.0):
        out, absout = oracle.attn_decode(q, k, v, scale=scale)
        e = math.exp(scale)
        w0, w1 = 1.0 / (1.0 + e), e / (1.0 + e)
        ref = [2.0 * w0 - 4.0 * w1, w1, -w0 + 3.0 * w1, 0.5]
        refabs = [2.0 * w0 + 4.0 * w1, w1, w0 + 3.0 * w1, 0.5]
        assert out.shape == (1, D)
        np.testing.assert_allclose(out[0], ref, rtol=1e-15, atol=1e-15)
        np.testing.assert_allclose(absout[0], refabs, rtol=1e-15, atol=1e-15)


def test_large_scores_do_not_overflow():
    # scores 1000 and 1001: exact weights 1/(1+e), e/(1+e) only if the max is subtracted.
    q = _bits([[1000.0, 0.0]])
    k = _bits([[1.0, 0.0], [1.0, 1.0]])
    q[0, 1] = _bits([1.0])[0]
    v = _bits([[1.0, 0.0], [0.0, 1.0]])
    out, _ = oracle.attn_decode(q, k, v, scale=1.0)
    e = math.e
    np.testing.assert_allclose(out[0], [1.0 / (1.0 + e), e / (1.0 + e)], rtol=1e-14)


@pytest.mark.parametrize("qpos,window", [(100, 0), (100, 30), (31, 30), (5, 512)])
def test_ring_mask_rules(qpos, window):
    """Kept = position >= 0, <= qpos, and > qpos - window (window > 0): boundaries
    exactly as in the listing; masked slots cannot influence the result."""
    T, D = 24, 16
    q = synth.gen_attn_q(13, 8, D)
    k, v = synth.gen_attn_kv(13, T, D)
    kpos = np.array([-1, qpos + 1, qpos, qpos - window, qpos - window + 1, qpos - 1, 0, -5]
                    + list(range(qpos - 16, qpos)), dtype=np.int32)
    keep = (kpos >= 0) & (kpos <= qpos) & ((window <= 0) | (kpos > qpos - window))
    out, absout = oracle.attn_decode(q, k, v, kpos, qpos=qpos, window=window, scale=0.25)
    # The same cache with the masked slots removed.
    out2, absout2 = oracle.attn_decode(q, k[keep], v[keep], kpos[keep], qpos=qpos, window=window, scale=0.25)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(absout, absout2)
    # And with garbage in the masked slots.
    k3, v3 = k.copy(), v.copy()
    k3[~keep] = _bits(np.full((int((~keep).sum()), D), 300.0))
    v3[~keep] = _bits(np.full((int((~keep).sum()), D), -7e3))
    out3, _ = oracle.attn_decode(q, k3, v3, kpos, qpos=qpos, window=window, scale=0.25)
    np.testing.assert_array_equal(out, out3)


def test_no_kept_slot_gives_zero():
    q = synth.gen_attn_q(14, 8, 16)
    k, v = synth.gen_attn_kv(14, 5, 16)
    out, absout = oracle.attn_decode(q, k, v, np.full(5, -1, np.int32), qpos=10)
    assert not out.any() and not absout.any()


def test_slot_permutation_invariance():
    q = synth.gen_attn_q(15, 8, 32)
    k, v = synth.gen_attn_kv(15, 64, 32)
    kpos = synth.ring_positions(200, 64)
    perm = np.random.default_rng(0).permutation(64)
    a, _ = oracle.attn_decode(q, k, v, kpos, qpos=200, window=50, scale=0.2)
    b, _ = oracle.attn_decode(q, k[perm], v[perm], kpos[perm], qpos=200, window=50, scale=0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_matches_library_softmax():
    """Special case through library routines: numpy float64 matmul + scipy softmax."""
    special = pytest.importorskip("scipy.special")
    H, T, D, scale = 8, 300, 64, 1.0 / 8.0
    q = synth.gen_attn_q(16, H, D)
    k, v = synth.gen_attn_kv(16, T, D)
    out, absout = oracle.attn_decode(q, k, v, scale=scale)
    s = scale * (_val(q) @ _val(k).T)
    w = special.softmax(s, axis=1)
    np.testing.assert_allclose(out, w @ _val(v), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(absout, w @ np.abs(_val(v)), rtol=1e-11, atol=1e-13)


def test_score_shift_invariance():
    """An extra dimension adding the same constant to every score changes nothing."""
    H, T, D = 8, 50, 15
    q = synth.gen_attn_q(17, H, D)
    k, v = synth.gen_attn_kv(17, T, D)
    base, _ = oracle.attn_decode(q, k, v, scale=1.0)
    q2 = np.concatenate([q, np.full((H, 1), _bits([3.0])[0], np.uint16)], axis=1)
    k2 = np.concatenate([k, np.full((T, 1), _bits([1.0])[0], np.uint16)], axis=1)
    v2 = np.concatenate([v, np.zeros((T, 1), np.uint16)], axis=1)
    shifted, _ = oracle.attn_decode(q2, k2, v2, scale=1.0)
    np.testing.assert_allclose(shifted[:, :D], base, rtol=1e-12, atol=1e-14)


def test_ring_positions_match_a_simulated_ring():
    for slots, qpos in [(8, 3), (8, 7), (8, 20), (512, 511), (512, 70000)]:
        ring = np.full(slots, -1, np.int64)
        start = max(0, qpos - 3 * slots)
        for p in range(start, qpos + 1):
            ring[p % slots] = p
        np.testing.assert_array_equal(synth.ring_positions(qpos, slots), ring)


def test_page_cache_sizes():
    """The head widths of the attention workloads reproduce the pages' byte counts:
    2 KiB per token per full layer (one head of width 512, keys and values in
    16 bits) and 774 MiB for 131,072 tokens with 3 full layers and 12 sliding
    512-slot rings (which fixes the sliding head width at 256)."""
    full = 2 * 512 * 2
    assert full == 2048
    sliding = 2 * 256 * 2
    total = 3 * 131072 * full + 12 * 512 * sliding
    assert total == 774 * 2 ** 20
