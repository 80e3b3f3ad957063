"""Seeded synthetic inputs for the W4A16 path (shared by the oracle tests and the CUDA path).

This module holds no arithmetic of the method itself: it only draws the data that
both sides consume. Every draw is counter-based, so any slice of a stream can be
regenerated without the rest.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014). Draw i of the stream with initial state s0 is
mix(s0 + (i+1) * 0x9E3779B97F4A7C15) with the published 64-bit finaliser.
Normals: Box-Muller (1958) in fp64 on pairs of 53-bit uniforms.

Distributions (the workload statement of the W4A16 GEMV configs):
  codes  : the low 32 bits of successive draws are whole uint32 words, so every
           4-bit code is uniform over 0..15.
  steps  : bf16(|N(0,1)| * 0.02 + 1e-4), one per group of 32 along K.
  x      : bf16(N(0,1)).
  ids    : uniform integers in [0, n_rows).
Rounding of generated values: fp64 -> fp32 (round to nearest even) -> bf16 (round
to nearest even). The bf16 bits are the data; both sides consume the same bits.

Stream state: seed * 0x9E3779B97F4A7C15 + tag (mod 2^64), with tag 0 = codes,
1 = steps, 2 = x (one row), 3 = ids, 4 = x (several rows), 5 = probe buffer,
6 = attention query, 7 = cached keys, 8 = cached values.

Attention inputs (decode attention over a one-head key/value cache): q, keys and
values bf16(N(0,1)); the ring of a sliding layer holds the last `slots` positions
up to the query's (slot j = position p with p % slots == j), empty slots -1.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TAG_CODES, TAG_STEPS, TAG_X, TAG_IDS, TAG_XROWS, TAG_PROBE = 0, 1, 2, 3, 4, 5
TAG_Q, TAG_K, TAG_V = 6, 7, 8

_CHUNK = 1 << 20
_S27, _S30, _S31 = np.uint64(27), np.uint64(30), np.uint64(31)


def stream_state(seed: int, tag: int) -> int:
    return (seed * 0x9E3779B97F4A7C15 + tag) & 0xFFFFFFFFFFFFFFFF


def splitmix64(state0: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the SplitMix64 stream with initial state state0."""
    out = np.empty(count, dtype=np.uint64)
    s0 = np.uint64(state0)
    n0 = min(_CHUNK, count)
    z = np.empty(n0, dtype=np.uint64)
    t = np.empty(n0, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for c0 in range(0, count, _CHUNK):
            n = min(_CHUNK, count - c0)
            zz, tt = z[:n], t[:n]
            zz[:] = np.arange(start + c0 + 1, start + c0 + 1 + n, dtype=np.uint64)
            np.multiply(zz, GOLDEN_GAMMA, out=zz)
            np.add(zz, s0, out=zz)
            np.right_shift(zz, _S30, out=tt)
            np.bitwise_xor(zz, tt, out=zz)
            np.multiply(zz, _M1, out=zz)
            np.right_shift(zz, _S27, out=tt)
            np.bitwise_xor(zz, tt, out=zz)
            np.multiply(zz, _M2, out=zz)
            np.right_shift(zz, _S31, out=tt)
            np.bitwise_xor(zz, tt, out=out[c0:c0 + n])
    return out


def uniform53(state0: int, start: int, count: int) -> np.ndarray:
    """fp64 uniforms in [0, 1): the top 53 bits of each draw times 2^-53."""
    return (splitmix64(state0, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(state0: int, count: int, start: int = 0) -> np.ndarray:
    """N(0,1) values start .. start+count-1 of a Box-Muller stream (fp64).

    Value 2j is r*cos(2*pi*u2) and value 2j+1 is r*sin(2*pi*u2) for the uniform
    pair (draw 2j, draw 2j+1), r = sqrt(-2 ln(1 - draw 2j)). start must be even.
    """
    assert start % 2 == 0
    pairs = (count + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    p_base = start // 2
    for p0 in range(0, pairs, _CHUNK):
        n = min(_CHUNK, pairs - p0)
        u = uniform53(state0, 2 * (p_base + p0), 2 * n)
        u1 = 1.0 - u[0::2]  # (0, 1], keeps log finite
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        out[2 * p0:2 * (p0 + n):2] = r * np.cos(t)
        out[2 * p0 + 1:2 * (p0 + n):2] = r * np.sin(t)
    return out[:count]


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE, numpy cast) -> bf16 bits (RNE). Finite inputs only."""
    u = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gen_qweight(seed: int, n: int, k: int) -> np.ndarray:
    """uint32 [n][k/8]: 8 codes per word, every nibble uniform 0..15."""
    assert k % 8 == 0
    w = splitmix64(stream_state(seed, TAG_CODES), 0, n * (k // 8))
    return (w & np.uint64(0xFFFFFFFF)).astype(np.uint32).reshape(n, k // 8)


def gen_scales(seed: int, n: int, k: int, group: int = 32) -> np.ndarray:
    """bf16 bits [n][k/group]: |N(0,1)| * 0.02 + 1e-4."""
    assert k % group == 0
    z = normals(stream_state(seed, TAG_STEPS), n * (k // group))
    return f64_to_bf16_bits(np.abs(z) * 0.02 + 1e-4).reshape(n, k // group)


def gen_qweight_rows(seed: int, n: int, k: int, rows) -> np.ndarray:
    """Rows `rows` of gen_qweight(seed, n, k) without drawing the whole table."""
    w = k // 8
    s = stream_state(seed, TAG_CODES)
    out = np.empty((len(rows), w), dtype=np.uint32)
    for i, r in enumerate(rows):
        assert 0 <= r < n
        out[i] = (splitmix64(s, int(r) * w, w) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return out


def gen_scales_rows(seed: int, n: int, k: int, rows, group: int = 32) -> np.ndarray:
    """Rows `rows` of gen_scales(seed, n, k, group) without drawing the whole table."""
    gpr = k // group
    s = stream_state(seed, TAG_STEPS)
    out = np.empty((len(rows), gpr), dtype=np.uint16)
    for i, r in enumerate(rows):
        assert 0 <= r < n
        start = int(r) * gpr
        lead = start % 2
        z = normals(s, gpr + lead, start - lead)[lead:]
        out[i] = f64_to_bf16_bits(np.abs(z) * 0.02 + 1e-4)
    return out


def gen_x(seed: int, m: int, k: int) -> np.ndarray:
    """bf16 bits [m][k], N(0,1). One row uses tag 2, several rows tag 4."""
    tag = TAG_X if m == 1 else TAG_XROWS
    return f64_to_bf16_bits(normals(stream_state(seed, tag), m * k)).reshape(m, k)


def gen_ids(seed: int, count: int, n_rows: int) -> np.ndarray:
    """int32 [count], uniform in [0, n_rows): (high 32 bits * n_rows) >> 32."""
    z = splitmix64(stream_state(seed, TAG_IDS), 0, count) >> np.uint64(32)
    return ((z * np.uint64(n_rows)) >> np.uint64(32)).astype(np.int32)


def gen_words(seed: int, nwords: int) -> np.ndarray:
    """uint32 [nwords] of uniform bits (buffer for the memory read probe)."""
    w = splitmix64(stream_state(seed, TAG_PROBE), 0, nwords)
    return (w & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def gen_attn_q(seed: int, heads: int, d: int) -> np.ndarray:
    """bf16 bits [heads][d], N(0,1)."""
    return f64_to_bf16_bits(normals(stream_state(seed, TAG_Q), heads * d)).reshape(heads, d)


def gen_attn_kv(seed: int, slots: int, d: int, start: int = 0):
    """(k, v) bf16 bits [slots][d], N(0,1); rows start .. start+slots-1 of the streams."""
    k = f64_to_bf16_bits(normals(stream_state(seed, TAG_K), slots * d, start * d)).reshape(slots, d)
    v = f64_to_bf16_bits(normals(stream_state(seed, TAG_V), slots * d, start * d)).reshape(slots, d)
    return k, v


def ring_positions(qpos: int, slots: int) -> np.ndarray:
    """int32 [slots]: the position each ring slot records after writing 0..qpos (-1 = empty)."""
    j = np.arange(slots, dtype=np.int64)
    p = qpos - ((qpos - j) % slots)
    return np.where(p >= 0, p, -1).astype(np.int32)


def gen_w4_problem(seed: int, m: int, n: int, k: int, group: int = 32):
    """(x bf16 [m][k], qweight u32 [n][k/8], scales bf16 [n][k/group]) for one projection."""
    return gen_x(seed, m, k), gen_qweight(seed, n, k), gen_scales(seed, n, k, group)


# ---------------------------------------------------------------------------
# Device-side copy of the integer streams (same bits as the numpy version).
# Large code tables (GB) are drawn on the GPU with torch int64 arithmetic, which
# wraps like uint64 for +, *, ^; the logical right shift is an arithmetic shift
# followed by a mask. Only integer streams are drawn this way: the fp64
# Box-Muller streams always come from numpy on the host.

def _s64(v: int) -> int:
    v &= 0xFFFFFFFFFFFFFFFF
    return v - (1 << 64) if v >= (1 << 63) else v


def splitmix64_torch(state0: int, start: int, count: int, device, chunk: int = 1 << 24):
    import torch
    out = torch.empty(count, dtype=torch.int64, device=device)
    g, m1, m2, s0 = _s64(0x9E3779B97F4A7C15), _s64(0xBF58476D1CE4E5B9), _s64(0x94D049BB133111EB), _s64(state0)
    for c0 in range(0, count, chunk):
        n = min(chunk, count - c0)
        z = torch.arange(start + c0 + 1, start + c0 + 1 + n, dtype=torch.int64, device=device)
        z.mul_(g).add_(s0)
        z.bitwise_xor_((z >> 30) & ((1 << 34) - 1))
        z.mul_(m1)
        z.bitwise_xor_((z >> 27) & ((1 << 37) - 1))
        z.mul_(m2)
        z.bitwise_xor_((z >> 31) & ((1 << 33) - 1))
        out[c0:c0 + n] = z
    return out


def gen_qweight_torch(seed: int, n: int, k: int, device, out=None):
    """Device int32 [n][k/8] with the same bits as gen_qweight(seed, n, k)."""
    import torch
    assert k % 8 == 0
    count = n * (k // 8)
    q = torch.empty(count, dtype=torch.int32, device=device) if out is None else out.view(-1)
    chunk = 1 << 24
    for c0 in range(0, count, chunk):
        c = min(chunk, count - c0)
        z = splitmix64_torch(stream_state(seed, TAG_CODES), c0, c, device)
        lo = z & 0xFFFFFFFF
        q[c0:c0 + c] = torch.where(lo >= (1 << 31), lo - (1 << 32), lo).to(torch.int32)
    return q.view(n, k // 8)
