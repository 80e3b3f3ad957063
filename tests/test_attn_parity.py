"""GPU parity of w4_attn_decode against the fp64 oracle (through the C ABI).

Tolerance (derived from the kernel's arithmetic, elementwise):
  |out - ref| <= attn_rel_bound(D, S, T) * sum_t w_t |v_t| + 1e-6
where w are the exact softmax weights (the oracle's absout is sum_t w_t |v_t|)
and S = max over kept slots of scale * sum_d |q_d k_d|; the terms are given in
_util.attn_rel_bound (weights applied as two bf16 parts, exp2, the fp32 score
sums, the fp32 accumulation chain).
"""
import numpy as np
import pytest

import oracle
import synth

from _util import attn_rel_bound, to_dev_bits16
from _guard import guarded

pytestmark = pytest.mark.gpu


def _w4():
    import bit_weight_only_w4a16_gb300 as w4
    return guarded(w4)


def _score_scale(q, k, keep, scale):
    qf = np.abs(synth.bf16_bits_to_f32(q).astype(np.float64))
    kf = np.abs(synth.bf16_bits_to_f32(k[keep]).astype(np.float64))
    if kf.shape[0] == 0:
        return 0.0
    return float(scale * (qf @ kf.T).max())


def _keep(kpos, T, qpos, window):
    p = np.arange(T) if kpos is None else kpos.astype(np.int64)
    return (p >= 0) & (p <= qpos) & ((window <= 0) | (p > qpos - window))


def _check(q, k, v, kpos, qpos, window, scale, what):
    import torch
    w4 = _w4()
    H, D = q.shape
    T = k.shape[0]
    kp_dev = None if kpos is None else torch.from_numpy(np.ascontiguousarray(kpos, np.int32)).cuda()
    out = w4.w4_attn_decode(to_dev_bits16(q), to_dev_bits16(k), to_dev_bits16(v), kp_dev, qpos=qpos,
                            window=window, scale=scale)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref, absout = oracle.attn_decode(q, k, v, kpos, qpos=qpos, window=window, scale=scale)
    S = _score_scale(q, k, _keep(kpos, T, qpos, window), scale)
    rel = attn_rel_bound(D, S, T)
    err = np.abs(got - ref)
    bound = rel * absout + 1e-6
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst ratio "
                           f"{(err / bound).max():.3f}")
    return got, float((err / np.maximum(absout, 1e-30)).max())


@pytest.mark.parametrize("H,T,D", [(8, 1, 512), (8, 17, 512), (8, 1000, 512), (8, 4096, 256), (1, 300, 128),
                                   (3, 777, 384), (8, 20000, 512)])
def test_full_cache_matches_oracle(H, T, D):
    q = synth.gen_attn_q(100 + T, H, D)
    k, v = synth.gen_attn_kv(100 + T, T, D)
    _check(q, k, v, None, T - 1, 0, 1.0 / np.sqrt(D), f"H={H} T={T} D={D}")


@pytest.mark.parametrize("qpos,window", [(700, 512), (100, 512), (5000, 200), (511, 512)])
def test_sliding_ring_matches_oracle(qpos, window):
    """The 512-slot ring of a sliding layer (head width 256), full and partly empty."""
    H, T, D = 8, 512, 256
    q = synth.gen_attn_q(300 + qpos, H, D)
    k, v = synth.gen_attn_kv(300 + qpos, T, D)
    kpos = synth.ring_positions(qpos, T)
    _check(q, k, v, kpos, qpos, window, 1.0 / 16.0, f"ring qpos={qpos} window={window}")


def test_masked_slots_are_never_read():
    """Empty and out-of-window slots hold NaN bits: the output must not see them."""
    H, T, D = 8, 512, 256
    q = synth.gen_attn_q(401, H, D)
    k, v = synth.gen_attn_kv(401, T, D)
    qpos, window = 300, 128
    kpos = synth.ring_positions(qpos, T)
    keep = _keep(kpos, T, qpos, window)
    k[~keep] = 0x7FC0
    v[~keep] = 0x7FC0
    got, _ = _check(q, k, v, kpos, qpos, window, 1.0 / 16.0, "NaN in masked slots")
    assert np.isfinite(got).all()


def test_no_kept_slot_gives_zero():
    import torch
    w4 = _w4()
    H, T, D = 8, 64, 128
    q = synth.gen_attn_q(402, H, D)
    k, v = synth.gen_attn_kv(402, T, D)
    kpos = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    out = w4.w4_attn_decode(to_dev_bits16(q), to_dev_bits16(k), to_dev_bits16(v), kpos, qpos=10)
    torch.cuda.synchronize()
    assert not out.cpu().numpy().any()


def test_deterministic_run_to_run():
    import torch
    w4 = _w4()
    H, T, D = 8, 9000, 512
    q, (k, v) = synth.gen_attn_q(403, H, D), synth.gen_attn_kv(403, T, D)
    qd, kd, vd = to_dev_bits16(q), to_dev_bits16(k), to_dev_bits16(v)
    a = w4.w4_attn_decode(qd, kd, vd, scale=0.05).cpu().numpy()
    b = w4.w4_attn_decode(qd, kd, vd, scale=0.05).cpu().numpy()
    np.testing.assert_array_equal(a, b)


def test_full_length_cache_131072():
    """The full-length layer at the pages' largest context: 131,072 slots, head width 512."""
    H, T, D = 8, 131072, 512
    q = synth.gen_attn_q(404, H, D)
    k, v = synth.gen_attn_kv(404, T, D)
    _check(q, k, v, None, T - 1, 0, 1.0 / np.sqrt(D), "T=131072")


def test_rejects_unsupported_shapes():
    import torch
    w4 = _w4()
    q = torch.zeros((9, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error):
        w4.w4_attn_decode(q, k, k)  # 9 query heads
    q = torch.zeros((8, 640), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((4, 640), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w4.W4Error):
        w4.w4_attn_decode(q, k, k)  # head width beyond 512
