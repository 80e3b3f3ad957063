"""GPU parity of the device-resident decode-step plumbing against the oracle
(through the C ABI): the key/value append at a device position, attention
reading its position from device memory, the greedy LM head with the
forced-token skip, the next-step prologue, and a decode loop replayed from one
captured CUDA graph.

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the CUDA-graph paragraph
(one captured step replayed for every token, every position on the GPU), the
cache paragraph (ring and full-length layers), the emb4 paragraph (embedding and
LM head share one 4-bit table) and the tool-calling paragraph (a forced token
skips the LM-head read).

Bars: appends, history, positions, status words and gathered rows bit-exact;
attention within the decode-attention bound (derived in test_attn_parity.py:
(2^-8 + 2 D 2^-23 S) * sum_t w_t |v_t| + 1e-6); logits within 1e-4 * sum|w x| +
1e-6; a greedy pick equal to the oracle's where the oracle's top two logits are
more than twice that apart, and otherwise within it of the largest logit.
"""
import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, attn_rel_bound, bits16, to_dev_bits16, to_dev_u32
from _guard import check_all, gempty, gfrom, gfull, guarded, gzeros

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


def _i32(v):
    return gfrom(np.atleast_1d(np.asarray(v, dtype=np.int32)))


def _attn_close(got, q, k, v, kpos, qpos, window, scale, what):
    ref, absout = oracle.attn_decode(q, k, v, kpos, qpos=qpos, window=window, scale=scale)
    T = k.shape[0]
    p = np.arange(T) if kpos is None else np.asarray(kpos, np.int64)
    keep = (p >= 0) & (p <= qpos) & ((window <= 0) | (p > qpos - window))
    S = 0.0
    if keep.any():
        qf = np.abs(synth.bf16_bits_to_f32(q).astype(np.float64))
        kf = np.abs(synth.bf16_bits_to_f32(k[keep]).astype(np.float64))
        S = float(scale * (qf @ kf.T).max())
    D = q.shape[1]
    bound = attn_rel_bound(D, S, T) * absout + 1e-6
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert (err <= bound).all(), f"{what}: worst ratio {(err / bound).max():.3f}"


# ------------------------------------------------------------ attention ----

@pytest.mark.parametrize("T,D,qpos,window,ring", [(512, 256, 700, 512, True), (512, 256, 100, 512, True),
                                                  (5000, 512, 4999, 0, False), (5000, 512, 1234, 0, False),
                                                  (5000, 512, 3000, 300, False), (5000, 512, 0, 0, False),
                                                  (300, 128, 40, 7, False)])
def test_device_position_matches_host_position(w4, T, D, qpos, window, ring):
    """The device-position call is bitwise the host-position call, and both match
    the oracle (full caches with the query before the last slot exercise the
    dropped empty tiles)."""
    import torch
    H = 8
    q = synth.gen_attn_q(910 + T + qpos, H, D)
    k, v = synth.gen_attn_kv(910 + T + qpos, T, D)
    kpos = synth.ring_positions(qpos, T) if ring else None
    qd, kd, vd = to_dev_bits16(q), to_dev_bits16(k), to_dev_bits16(v)
    kp = None if kpos is None else torch.from_numpy(kpos).cuda()
    scale = D ** -0.5
    a = w4.w4_attn_decode(qd, kd, vd, kp, qpos=qpos, window=window, scale=scale)
    b = w4.w4_attn_decode(qd, kd, vd, kp, qpos=_i32(qpos), window=window, scale=scale)
    torch.cuda.synchronize()
    a, b = a.cpu().numpy(), b.cpu().numpy()
    np.testing.assert_array_equal(a, b)
    _attn_close(a, q, k, v, kpos, qpos, window, scale, f"T={T} qpos={qpos} window={window}")


def test_masked_tail_of_full_cache_is_never_read(w4):
    """Slots after the query position hold NaN bits; the dropped tiles and the
    masks keep them out of the result."""
    import torch
    H, T, D, qpos = 8, 4096, 256, 1000
    q = synth.gen_attn_q(930, H, D)
    k, v = synth.gen_attn_kv(930, T, D)
    k[qpos + 1:] = 0x7FC0
    v[qpos + 1:] = 0x7FC0
    out = w4.w4_attn_decode(to_dev_bits16(q), to_dev_bits16(k), to_dev_bits16(v), qpos=_i32(qpos), scale=0.06)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    _attn_close(got, q, k, v, None, qpos, 0, 0.06, "NaN tail")


# ---------------------------------------------------------------- append ----

@pytest.mark.parametrize("T,D,P", [(16, 128, 41), (5, 72, 13)])
def test_kv_append_ring_and_full_cache(w4, T, D, P):
    import torch
    kall, vall = synth.gen_attn_kv(940, P, D)
    kr = gzeros((T, D), torch.int16)
    vr = gzeros((T, D), torch.int16)
    kp = gfull((T,), -1, torch.int32)
    kf = gzeros((T, D), torch.int16)
    vf = gzeros((T, D), torch.int16)
    pos = _i32(0)
    status = _i32(0)
    kro, vro, kpo = np.zeros((T, D), np.uint16), np.zeros((T, D), np.uint16), np.full(T, -1, np.int32)
    kfo, vfo = np.zeros((T, D), np.uint16), np.zeros((T, D), np.uint16)
    kd, vd = to_dev_bits16(kall), to_dev_bits16(vall)
    for p in range(P):
        pos.fill_(p)
        w4.w4_kv_append(kr, vr, kd[p], vd[p], pos, kpos=kp, status=status)
        w4.w4_kv_append(kf, vf, kd[p], vd[p], pos, status=status)
        kro, vro, kpo, _ = oracle.kv_append(kro, vro, kpo, kall[p], vall[p], p)
        kfo, vfo, _, sto = oracle.kv_append(kfo, vfo, None, kall[p], vall[p], p)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits16(kr), kro)
        np.testing.assert_array_equal(bits16(vr), vro)
        np.testing.assert_array_equal(kp.cpu().numpy(), kpo)
        np.testing.assert_array_equal(bits16(kf), kfo)
        np.testing.assert_array_equal(bits16(vf), vfo)
        assert int(status.item()) == sto  # the full cache overflows from position 16 on
        status.zero_()
    assert int(pos.item()) == P - 1  # the append never moves the position
    status.zero_()
    pos.fill_(-3)
    before = bits16(kr).copy()
    w4.w4_kv_append(kr, vr, kd[0], vd[0], pos, kpos=kp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    np.testing.assert_array_equal(bits16(kr), before)


# --------------------------------------------------------------- LM head ----

@pytest.mark.parametrize("N,K,group", [(4096, 1536, 32), (131072, 1536, 256), (1000, 512, 64)])
def test_forced_lm_head(w4, N, K, group):
    import torch
    x = synth.gen_x(950 + N, 1, K)
    qw = synth.gen_qweight(950 + N, N, K)
    sc = synth.gen_scales(950 + N, N, K, group)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    forced = _i32(-1)
    y, a = w4.w4a16_gemv_argmax_forced(xd, qd, sd, forced, group=group)
    y2, a2 = w4.w4a16_gemv_argmax_noalloc(xd, qd, sd, group=group)
    torch.cuda.synchronize()
    y, a = y.cpu().numpy(), int(a.item())
    np.testing.assert_array_equal(y, y2.cpu().numpy())  # the same kernels as the plain greedy call
    assert a == int(a2.cpu().numpy()[0])
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y, yr, ar, what=f"forced LM head (none) N={N}")
    idx, gap = oracle.argmax(yr[0])
    assert gap > 2 * (1e-4 * ar[0, idx] + 1e-6), "ambiguous seed"
    assert a == idx
    # Forced: argmax = the forced token, y untouched.
    yt = gfull((1, N), 12345.0, torch.float32)
    forced.fill_(N - 3)
    _, a3 = w4.w4a16_gemv_argmax_forced(xd, qd, sd, forced, group=group, out=yt)
    torch.cuda.synchronize()
    assert int(a3.item()) == N - 3
    assert (yt.cpu().numpy() == 12345.0).all()
    assert w4.device_error() == 0


# -------------------------------------------------------------- prologue ----

@pytest.mark.parametrize("group", [64, 512])
def test_prologue_bit_exact(w4, group):
    import torch
    V, K = 1000, 1536
    qt = synth.gen_qweight(960, V, K)
    sc = synth.gen_scales(960, V, K, group)
    qd, sd = to_dev_u32(qt), to_dev_bits16(sc)
    tokens = gfull((10,), -1, torch.int32)
    hist = np.full(10, -1, np.int32)
    pos, status = _i32(5), _i32(0)
    x = gempty((1, K), torch.bfloat16)
    cases = [(437, 0), (V, 1), (0, 0), (V - 1, 0), (-2, 1)]  # (token, expected new status bits)
    p = 5
    st_all = 0
    for tok, _ in cases:
        tk = _i32(tok)
        w4.w4_decode_prologue(tk, pos, qd, sd, group=group, x_next=x, tokens=tokens, status=status)
        xo, hist, p, st = oracle.decode_prologue(tok, p, hist, qt, sc, group)
        st_all |= st
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits16(x), xo)
        np.testing.assert_array_equal(tokens.cpu().numpy(), hist)
        assert int(pos.item()) == p
        assert int(status.item()) == st_all
    # p is now 10: the next token's index 11 lies outside the 10-entry history
    w4.w4_decode_prologue(_i32(3), pos, qd, sd, group=group, x_next=x, tokens=tokens, status=status)
    xo, hist2, p, st = oracle.decode_prologue(3, p, hist, qt, sc, group)
    torch.cuda.synchronize()
    assert st == 2 and int(status.item()) == st_all | 2
    np.testing.assert_array_equal(tokens.cpu().numpy(), hist2)
    np.testing.assert_array_equal(bits16(x), xo)


# ------------------------------------------------- graph-replayed loop ----

@pytest.mark.parametrize("tied", [False, True])
def test_graph_replayed_decode_loop(w4, tied):
    """150 decode steps replayed from ONE captured graph: append (ring of 64 slots
    and a full cache), attention at the device position for both, the LM head
    (every third token forced), prologue. Positions, history and x never leave
    the device; per-step host work is two row copies and the forced token.
    tied: the embedding and the LM head are one table (the emb4 paragraph)."""
    import torch
    S, H, D, Tr, Tf = 150, 8, 256, 64, 256
    V, K, group = 4096, 1536, 64
    scale = D ** -0.5
    q = synth.gen_attn_q(970, H, D)
    kall, vall = synth.gen_attn_kv(971, S, D)
    eq, es = synth.gen_qweight(972, V, K), synth.gen_scales(972, V, K, group)
    hq, hs = (eq, es) if tied else (synth.gen_qweight(973, V, K), synth.gen_scales(973, V, K, group))
    forced_seq = np.array([(s * 7919) % V if s % 3 == 1 else -1 for s in range(S)], np.int32)
    start = 17

    dev = torch.device("cuda")
    qd, kall_d, vall_d = to_dev_bits16(q), to_dev_bits16(kall), to_dev_bits16(vall)
    eqd, esd = to_dev_u32(eq), to_dev_bits16(es)
    hqd, hsd = (eqd, esd) if tied else (to_dev_u32(hq), to_dev_bits16(hs))
    forced_d = torch.from_numpy(forced_seq).to(dev)
    kr = gzeros((Tr, D), torch.int16)
    vr = gzeros((Tr, D), torch.int16)
    kpr = gfull((Tr,), -1, torch.int32)
    kf = gzeros((Tf, D), torch.int16)
    vf = gzeros((Tf, D), torch.int16)
    pos = gzeros((1,), torch.int32)
    knew = gempty((D,), torch.int16)
    vnew = gempty((D,), torch.int16)
    forced = gfull((1,), -1, torch.int32)
    y = gempty((1, V), torch.float32)
    am = gempty((1,), torch.int32)
    tokens = gfull((S + 1,), -1, torch.int32)
    status = gzeros((1,), torch.int32)
    att_r = gempty((H, D), torch.float32)
    att_f = gempty((H, D), torch.float32)
    x = gempty((1, K), torch.bfloat16)
    stream = torch.cuda.Stream()

    def step():
        w4.w4_kv_append(kr, vr, knew, vnew, pos, kpos=kpr, status=status, stream=stream)
        w4.w4_kv_append(kf, vf, knew, vnew, pos, status=status, stream=stream)
        w4.w4_attn_decode(qd, kr, vr, kpr, qpos=pos, window=Tr, scale=scale, out=att_r, stream=stream)
        w4.w4_attn_decode(qd, kf, vf, None, qpos=pos, scale=scale, out=att_f, stream=stream)
        w4.w4a16_gemv_argmax_forced(x, hqd, hsd, forced, group=group, out=y, argmax=am, stream=stream)
        w4.w4_decode_prologue(am, pos, eqd, esd, group=group, x_next=x, tokens=tokens, status=status,
                              stream=stream)

    def reset():
        kr.zero_(); vr.zero_(); kpr.fill_(-1); kf.zero_(); vf.zero_()
        pos.zero_(); tokens.fill_(-1); status.zero_(); forced.fill_(-1)
        tokens[0] = start
        w4.w4_embed_gather(tokens[:1], eqd, esd, group=group, out=x, stream=stream)

    with torch.cuda.stream(stream):
        knew.copy_(kall_d[0]); vnew.copy_(vall_d[0])
        reset()
        step()  # eager warm-up (first-call set-up outside the capture)
        reset()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    hist_r = torch.empty((S, H, D), dtype=torch.float32, device=dev)
    hist_f = torch.empty_like(hist_r)
    with torch.cuda.stream(stream):
        for s in range(S):
            knew.copy_(kall_d[s]); vnew.copy_(vall_d[s]); forced.copy_(forced_d[s:s + 1])
            g.replay()
            hist_r[s].copy_(att_r); hist_f[s].copy_(att_f)
    torch.cuda.synchronize()
    check_all("graph-replayed decode loop")
    got_tokens = tokens.cpu().numpy()
    got_r, got_f = hist_r.cpu().numpy(), hist_f.cpu().numpy()
    assert int(pos.item()) == S
    assert int(status.item()) == 0
    assert w4.device_error() == 0

    # The oracle, step by step; an ambiguous greedy pick follows the device's.
    kro, vro, kpo = np.zeros((Tr, D), np.uint16), np.zeros((Tr, D), np.uint16), np.full(Tr, -1, np.int32)
    kfo, vfo = np.zeros((Tf, D), np.uint16), np.zeros((Tf, D), np.uint16)
    hist = np.full(S + 1, -1, np.int32)
    hist[0] = start
    xo, _ = oracle.embed_gather(np.array([start], np.int32), eq, es, group)
    ambiguous = 0
    for s in range(S):
        kro, vro, kpo, st = oracle.kv_append(kro, vro, kpo, kall[s], vall[s], s)
        kfo, vfo, _, st2 = oracle.kv_append(kfo, vfo, None, kall[s], vall[s], s)
        assert st == 0 and st2 == 0
        _attn_close(got_r[s], q, kro, vro, kpo, s, Tr, scale, f"ring step {s}")
        _attn_close(got_f[s], q, kfo, vfo, None, s, 0, scale, f"full step {s}")
        tok, yr, ar = oracle.lm_head_pick(xo, hq, hs, group, int(forced_seq[s]))
        dev_tok = int(got_tokens[s + 1])
        if yr is not None:
            idx, gap = oracle.argmax(yr[0])
            tol = 1e-4 * ar[0] + 1e-6
            if gap > 2 * tol[idx]:
                assert dev_tok == idx, f"step {s}: device picked {dev_tok}, oracle {idx}"
            else:
                ambiguous += 1
                assert yr[0, dev_tok] >= yr[0, idx] - tol[idx] - tol[dev_tok], f"step {s}: invalid pick"
                tok = dev_tok
        xo, hist, p, st = oracle.decode_prologue(tok, s, hist, eq, es, group)
        assert st == 0 and p == s + 1
    np.testing.assert_array_equal(got_tokens, hist)
    np.testing.assert_array_equal(bits16(x), xo)
    assert ambiguous <= 5, ambiguous
