"""ctypes front end of the plain C oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this package. The CUDA library and its Python binding never do.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB = os.path.join(_HERE, "libw4a16_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host-only, portable C, no -march flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.w4o_gemm_rows.argtypes = [P, P, P, P, P, I, I, I, I, P, I]
        lib.w4o_gemm_rows.restype = None
        lib.w4o_dequant_rows.argtypes = [P, P, P, I, I, I, P, I]
        lib.w4o_dequant_rows.restype = None
        lib.w4o_argmax.argtypes = [P, I, P]
        lib.w4o_argmax.restype = I
        lib.w4o_embed_gather.argtypes = [P, P, P, P, I, I, I, I, P]
        lib.w4o_embed_gather.restype = None
        lib.w4o_sum_words.argtypes = [P, I]
        lib.w4o_sum_words.restype = ctypes.c_uint64
        lib.w4o_hadamard_rows.argtypes = [P, P, I, I, I]
        lib.w4o_hadamard_rows.restype = None
        lib.w4o_gemm_rows_xf64.argtypes = [P, P, P, P, P, I, I, I, I, P, I]
        lib.w4o_gemm_rows_xf64.restype = None
        lib.w4o_attn_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, ctypes.c_double, P]
        lib.w4o_attn_decode.restype = None
        lib.w4o_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.w4o_f32_to_bf16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def gemm(x, qweight, scales, group: int = 32, rows=None):
    """(y, absy) in fp64. x bf16 bits [M][K]; qweight u32 [N][K/8]; scales bf16 bits [N][K/g].

    rows: optional list of output rows to compute (then y is [M][len(rows)]).
    """
    lib = _load()
    x = _c(np.atleast_2d(x), np.uint16)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    M, K = x.shape
    N = qweight.shape[0]
    assert qweight.shape[1] * 8 == K and scales.shape == (N, K // group)
    if rows is None:
        r = None
        nr = N
    else:
        r = _c(rows, np.int64)
        nr = r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    a = np.empty((M, nr), dtype=np.float64)
    lib.w4o_gemm_rows(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales),
                      M, N, K, group, None if r is None else _ptr(r), nr)
    return y, a


def dequant(qweight, scales, group: int = 32, rows=None):
    lib = _load()
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    N, K = qweight.shape[0], qweight.shape[1] * 8
    r = None if rows is None else _c(rows, np.int64)
    nr = N if r is None else r.shape[0]
    w = np.empty((nr, K), dtype=np.float64)
    lib.w4o_dequant_rows(_ptr(w), _ptr(qweight), _ptr(scales), N, K, group,
                         None if r is None else _ptr(r), nr)
    return w


def argmax(y):
    """(index, gap) of a 1-D fp64 vector: lowest index of the max, -0 == +0."""
    lib = _load()
    y = _c(y, np.float64).ravel()
    gap = np.zeros(1, dtype=np.float64)
    idx = lib.w4o_argmax(_ptr(y), y.shape[0], _ptr(gap))
    return int(idx), float(gap[0])


def embed_gather(ids, qtable, scales, group: int = 32):
    """(out bf16 bits [M][K], flag) for the 4-bit row gather."""
    lib = _load()
    ids = _c(ids, np.int32).ravel()
    qtable = _c(qtable, np.uint32)
    scales = _c(scales, np.uint16)
    N, K = qtable.shape[0], qtable.shape[1] * 8
    out = np.empty((ids.shape[0], K), dtype=np.uint16)
    flag = np.zeros(1, dtype=np.int32)
    lib.w4o_embed_gather(_ptr(out), _ptr(ids), _ptr(qtable), _ptr(scales),
                         ids.shape[0], N, K, group, _ptr(flag))
    return out, int(flag[0])


def sum_words(buf):
    """Sum of the uint32 words of buf, mod 2^64."""
    lib = _load()
    b = _c(buf, np.uint32).ravel()
    return int(lib.w4o_sum_words(_ptr(b), b.shape[0]))


def f32_to_bf16(f: float) -> int:
    return int(_load().w4o_f32_to_bf16(float(f)))


def attn_decode(q, k, v, kpos=None, qpos=None, window: int = 0, scale: float = 1.0):
    """(out, absout) fp64 [H][D]: softmax(scale * q k^T) v over the kept cache slots.

    q bf16 bits [H][D]; k, v bf16 bits [T][D]; kpos int32 [T] (recorded position
    of each slot, -1 = empty) or None (slot t holds position t); qpos defaults to
    T - 1. absout is sum_t w_t |v_t|, the scale of the parity tolerance.
    """
    lib = _load()
    q = _c(np.atleast_2d(q), np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    H, D = q.shape
    T = k.shape[0]
    assert k.shape == (T, D) and v.shape == (T, D)
    kp = None if kpos is None else _c(kpos, np.int32).ravel()
    assert kp is None or kp.shape[0] == T
    qp = T - 1 if qpos is None else int(qpos)
    out = np.empty((H, D), dtype=np.float64)
    absout = np.empty((H, D), dtype=np.float64)
    s = np.empty(max(T, 1), dtype=np.float64)
    lib.w4o_attn_decode(_ptr(out), _ptr(absout), _ptr(q), _ptr(k), _ptr(v),
                        None if kp is None else _ptr(kp), qp, int(window), H, T, D, float(scale), _ptr(s))
    return out, absout


def hadamard(x, b: int):
    """fp64 [M][K]: x (bf16 bits) times blockdiag(H_b) with H_b[i][j] = (-1)^popcount(i&j)/sqrt(b)."""
    lib = _load()
    x = _c(np.atleast_2d(x), np.uint16)
    M, K = x.shape
    assert b >= 1 and (b & (b - 1)) == 0 and K % b == 0
    out = np.empty((M, K), dtype=np.float64)
    lib.w4o_hadamard_rows(_ptr(out), _ptr(x), M, K, b)
    return out


def gemm_xf64(x, qweight, scales, group: int = 32, rows=None):
    """gemm() with an fp64 activation [M][K] (e.g. hadamard(x, b))."""
    lib = _load()
    x = _c(np.atleast_2d(x), np.float64)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    M, K = x.shape
    N = qweight.shape[0]
    assert qweight.shape[1] * 8 == K and scales.shape == (N, K // group)
    r = None if rows is None else _c(rows, np.int64)
    nr = N if r is None else r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    a = np.empty((M, nr), dtype=np.float64)
    lib.w4o_gemm_rows_xf64(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K, group,
                           None if r is None else _ptr(r), nr)
    return y, a


def gemm_hadamard(x, qweight, scales, hblock: int, group: int = 32, rows=None):
    """(y, absy): the rotated product (x H) W'^T with W' = dequant(qweight, scales)."""
    return gemm_xf64(hadamard(x, hblock), qweight, scales, group, rows)


# ----------------------------------------------------------------------------
# Device-resident decode-step plumbing (reading R18). Sources: "Gemma 4 E2B on a
# 4 GB GPU with pure PyTorch" - the cache paragraph (full layers: one slot per
# position; sliding layers: a ring of slots recording each slot's position), the
# CUDA-graph paragraph (every position kept on the GPU so that one captured step
# replays for every token), the emb4 paragraph (embedding and LM head share one
# 4-bit table) and the tool-calling paragraph (a step whose constrained decoder
# admits one token skips the LM-head read).
#
# R18: the token at position p appends its key/value rows to slot p mod T of a
# ring (which records p) or slot p of a full cache before its attention runs;
# the step's LM head yields the token at position p + 1, either the greedy pick
# or the forced token (then no logits are formed); the prologue records it in
# the history at index p + 1, advances the position to p + 1 and looks up its
# embedding row (the plain 4-bit gather, no model-specific scaling).
# ----------------------------------------------------------------------------

def kv_append(k_cache, v_cache, kpos, k_new, v_new, pos: int):
    """(k_cache', v_cache', kpos', status) after appending position `pos`.

    kpos int32 [T] (ring) or None (full cache). Ring: slot pos mod T, whose
    recorded position becomes pos. Full cache: slot pos, which must lie in
    [0, T). A negative position, or one outside a full cache, changes nothing
    and gives status 1.
    """
    k_cache = np.array(k_cache, dtype=np.uint16, copy=True)
    v_cache = np.array(v_cache, dtype=np.uint16, copy=True)
    kp = None if kpos is None else np.array(kpos, dtype=np.int32, copy=True)
    T = k_cache.shape[0]
    pos = int(pos)
    if pos < 0 or (kp is None and pos >= T):
        return k_cache, v_cache, kp, 1
    slot = pos % T if kp is not None else pos
    k_cache[slot] = np.asarray(k_new, dtype=np.uint16).ravel()
    v_cache[slot] = np.asarray(v_new, dtype=np.uint16).ravel()
    if kp is not None:
        kp[slot] = pos
    return k_cache, v_cache, kp, 0


def lm_head_pick(x, qweight, scales, group: int, forced: int):
    """(token, y, absy): the forced token when forced >= 0 (y, absy None: no logits
    are formed), else the greedy pick, the lowest index of the largest logit of
    the one x-row (y, absy from gemm())."""
    if int(forced) >= 0:
        return int(forced), None, None
    y, a = gemm(x, qweight, scales, group)
    return argmax(y[0])[0], y, a


def decode_prologue(token: int, pos: int, tokens, qtable, scales, group: int = 32):
    """(x_next bf16 bits [1][K], tokens', pos + 1, status) of the next-step prologue.

    tokens: int32 history (or None); the token is stored at index pos + 1 when
    that index lies inside it (else status bit 1). A token outside the table
    gives a zero row and status bit 0 (the gather's own rule).
    """
    status = 0
    tk = None if tokens is None else np.array(tokens, dtype=np.int32, copy=True)
    nx = int(pos) + 1
    if tk is not None:
        if 0 <= nx < tk.shape[0]:
            tk[nx] = int(token)
        else:
            status |= 2
    row, flag = embed_gather(np.array([int(token)], dtype=np.int32), qtable, scales, group)
    if flag:
        status |= 1
    return row, tk, nx, status
