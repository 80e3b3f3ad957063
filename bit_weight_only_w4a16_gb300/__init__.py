"""Python binding of libw4a16.so, the W4A16 GEMV/GEMM library for GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/w4a16.h. Tensors must be CUDA
tensors on the current device; bf16 data may be passed either as torch.bfloat16
or as raw int16/uint16 bits. There is no CPU path: if the compiled library is
missing, importing the binding raises.

Weight format: qweight uint32 [N][K/8] (8 codes per word along K, low nibble
first, zero point 8), scales bf16 [N][K/32], x bf16 [M][K], y fp32 [M][N].
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

W4_OK = 0
STATUS_NAMES = {0: "W4_OK", 1: "W4_ERR_INVALID_ARG", 2: "W4_ERR_UNSUPPORTED",
                3: "W4_ERR_MISALIGNED", 4: "W4_ERR_CUDA", 5: "W4_ERR_NO_DEVICE"}

# Symbols declared in include/w4a16.h.
EXPORTS = ("w4_status_string", "w4_last_cuda_error", "w4_init", "w4_device_error", "w4a16_gemv", "w4a16_gemm",
           "w4a16_gemv_argmax", "w4a16_gemv_argmax_noalloc", "w4_embed_gather", "hbm_read_probe",
           "w4_attn_decode", "w4a16_gemv_hadamard", "w4_selftest_wait_timeout", "w4_attn_decode_devpos",
           "w4_kv_append", "w4a16_gemv_argmax_forced", "w4_decode_prologue")


class W4Error(RuntimeError):
    def __init__(self, status: int, call: str, detail: str = ""):
        self.status = status
        super().__init__(f"{call} -> {STATUS_NAMES.get(status, status)}" + (f" ({detail})" if detail else ""))


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with bit_weight_only_w4a16_gb300.build.build() "
                          "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4_status_string.argtypes = [I]
    lib.w4_status_string.restype = ctypes.c_char_p
    lib.w4_last_cuda_error.argtypes = []
    lib.w4_last_cuda_error.restype = ctypes.c_char_p
    lib.w4_init.argtypes = []
    lib.w4_init.restype = I
    lib.w4_device_error.argtypes = [P]
    lib.w4_device_error.restype = I
    for name in ("w4a16_gemv", "w4a16_gemm"):
        f = getattr(lib, name)
        f.argtypes = [P, P, P, P, I, I, I, I, P]
        f.restype = I
    for name in ("w4a16_gemv_argmax", "w4a16_gemv_argmax_noalloc"):
        f = getattr(lib, name)
        f.argtypes = [P, P, P, P, P, I, I, I, I, P]
        f.restype = I
    lib.w4_embed_gather.argtypes = [P, P, P, P, I, I, I, I, P, P]
    lib.w4_embed_gather.restype = I
    lib.hbm_read_probe.argtypes = [P, P, S, P]
    lib.hbm_read_probe.restype = I
    lib.w4_attn_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_float, P]
    lib.w4_attn_decode.restype = I
    lib.w4a16_gemv_hadamard.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
    lib.w4a16_gemv_hadamard.restype = I
    lib.w4_selftest_wait_timeout.argtypes = [P]
    lib.w4_selftest_wait_timeout.restype = I
    lib.w4_attn_decode_devpos.argtypes = [P, P, P, P, P, P, I, I, I, I, ctypes.c_float, P]
    lib.w4_attn_decode_devpos.restype = I
    lib.w4_kv_append.argtypes = [P, P, P, P, P, P, I, I, P, P]
    lib.w4_kv_append.restype = I
    lib.w4a16_gemv_argmax_forced.argtypes = [P, P, P, P, P, I, I, I, P, P]
    lib.w4a16_gemv_argmax_forced.restype = I
    lib.w4_decode_prologue.argtypes = [P, P, P, P, P, P, I, I, I, I, P, P]
    lib.w4_decode_prologue.restype = I
    return lib


_lib = load_library()


def _check(rc: int, call: str):
    if rc != W4_OK:
        detail = _lib.w4_last_cuda_error().decode() if rc == 4 else ""
        raise W4Error(rc, call, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _bits16(t, name):
    _cuda(t, name)
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bf16 (or its raw 16-bit bits)")
    return t


def _u32(t, name):
    _cuda(t, name)
    if t.dtype not in (torch.int32, torch.uint32):
        raise TypeError(f"{name} must be a 32-bit integer tensor of packed words")
    return t


def init():
    """Set up the library on the current device (call before CUDA graph capture)."""
    _check(_lib.w4_init(), "w4_init")


def device_error() -> int:
    """Synchronize the device, then read and clear the library's device error word."""
    code = ctypes.c_int32(0)
    _check(_lib.w4_device_error(ctypes.byref(code)), "w4_device_error")
    return int(code.value)


def _shape(x, qweight, scales, group):
    M, K = x.shape
    N = qweight.shape[0]
    if qweight.shape[1] * 8 != K or tuple(scales.shape) != (N, K // group):
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, qweight {tuple(qweight.shape)}, "
                         f"scales {tuple(scales.shape)}")
    return M, N, K


def w4a16_gemv(x, qweight, scales, group: int = 32, out=None, stream=None):
    """y[M][N] fp32 = x[M][K] @ dequant(qweight, scales)^T for M <= 8 (decode)."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    M, N, K = _shape(x, qweight, scales, group)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    _check(_lib.w4a16_gemv(_ptr(y), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K, group,
                           _stream(stream)), "w4a16_gemv")
    return y


def w4a16_gemm(x, qweight, scales, group: int = 32, out=None, stream=None):
    """y[M][N] fp32 for any M (M > 8 runs the tensor-core prefill kernel)."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    M, N, K = _shape(x, qweight, scales, group)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    _check(_lib.w4a16_gemm(_ptr(y), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K, group,
                           _stream(stream)), "w4a16_gemm")
    return y


def w4a16_gemv_argmax(x, qweight, scales, group: int = 32, out=None, argmax=None, stream=None):
    """(y fp32 [M][N], argmax int32 [M]): decode GEMV with the greedy pick fused."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    M, N, K = _shape(x, qweight, scales, group)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    a = torch.empty((M,), dtype=torch.int32, device=x.device) if argmax is None else _cuda(argmax, "argmax")
    _check(_lib.w4a16_gemv_argmax(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K,
                                  group, _stream(stream)), "w4a16_gemv_argmax")
    return y, a


def w4a16_gemv_argmax_noalloc(x, qweight, scales, group: int = 32, out=None, argmax=None, stream=None):
    """w4a16_gemv_argmax whose library scratch is a fixed device array (no device
    allocation inside the call; y and argmax are allocated here only when the
    caller does not pass them)."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    M, N, K = _shape(x, qweight, scales, group)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    a = torch.empty((M,), dtype=torch.int32, device=x.device) if argmax is None else _cuda(argmax, "argmax")
    _check(_lib.w4a16_gemv_argmax_noalloc(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K,
                                          group, _stream(stream)), "w4a16_gemv_argmax_noalloc")
    return y, a


def w4_embed_gather(ids, qtable, scales, group: int = 32, out=None, status=None, stream=None):
    """bf16 [M][K] rows of the 4-bit table for int32 ids [M] (raw bits as int16)."""
    _cuda(ids, "ids"); _u32(qtable, "qtable"); _bits16(scales, "scales")
    if ids.dtype != torch.int32:
        raise TypeError("ids must be int32")
    M = ids.numel()
    N, K = qtable.shape[0], qtable.shape[1] * 8
    if tuple(scales.shape) != (N, K // group):
        raise ValueError("scales shape mismatch")
    o = torch.empty((M, K), dtype=torch.bfloat16, device=ids.device) if out is None else _cuda(out, "out")
    _check(_lib.w4_embed_gather(_ptr(o), _ptr(ids), _ptr(qtable), _ptr(scales), M, N, K, group,
                                _ptr(status), _stream(stream)), "w4_embed_gather")
    return o


def hbm_read_probe(buf, out=None, stream=None):
    """Device uint64 (as int64) sum of buf's uint32 words mod 2^64 (one streaming read)."""
    _cuda(buf, "buf")
    nbytes = buf.numel() * buf.element_size()
    s = torch.empty((1,), dtype=torch.int64, device=buf.device) if out is None else _cuda(out, "out")
    _check(_lib.hbm_read_probe(_ptr(s), _ptr(buf), nbytes, _stream(stream)), "hbm_read_probe")
    return s


def w4_attn_decode(q, k, v, kpos=None, qpos=None, window: int = 0, scale: float = 1.0, out=None, stream=None):
    """fp32 [H][D]: softmax(scale * q k^T) v over the kept slots of a one-head cache.

    q bf16 [H][D] (H <= 8 query heads sharing the key/value head); k, v bf16 [T][D];
    kpos int32 [T] (position recorded in each slot, -1 = empty) or None (slot t
    holds position t); qpos defaults to T - 1, or is a device int32 [1] tensor read
    when the kernels run (w4_attn_decode_devpos); window 0 = no window.
    """
    _bits16(q, "q"); _bits16(k, "k"); _bits16(v, "v")
    H, D = q.shape
    T = k.shape[0]
    if tuple(k.shape) != (T, D) or tuple(v.shape) != (T, D):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if kpos is not None:
        _cuda(kpos, "kpos")
        if kpos.dtype != torch.int32 or kpos.numel() != T:
            raise ValueError("kpos must be int32 [T]")
    o = torch.empty((H, D), dtype=torch.float32, device=q.device) if out is None else _cuda(out, "out")
    if isinstance(qpos, torch.Tensor):
        _cuda(qpos, "qpos")
        if qpos.dtype != torch.int32 or qpos.numel() != 1:
            raise ValueError("a device qpos must be int32 [1]")
        _check(_lib.w4_attn_decode_devpos(_ptr(o), _ptr(q), _ptr(k), _ptr(v), _ptr(kpos), _ptr(qpos), int(window),
                                          H, T, D, float(scale), _stream(stream)), "w4_attn_decode_devpos")
        return o
    qp = T - 1 if qpos is None else int(qpos)
    _check(_lib.w4_attn_decode(_ptr(o), _ptr(q), _ptr(k), _ptr(v), _ptr(kpos), qp, int(window), H, T, D,
                               float(scale), _stream(stream)), "w4_attn_decode")
    return o


def w4a16_gemv_hadamard(x, qweight, scales, hblock: int, group: int = 32, out=None, argmax=False,
                        stream=None):
    """y fp32 [M][N] = (x H) W'^T for Hadamard-rotated weights W' (M <= 4); with
    argmax=True (or an int32 [M] tensor) also the lowest index of each row's max."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    M, N, K = _shape(x, qweight, scales, group)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    a = None
    if argmax is True:
        a = torch.empty((M,), dtype=torch.int32, device=x.device)
    elif argmax is not False and argmax is not None:
        a = _cuda(argmax, "argmax")
    _check(_lib.w4a16_gemv_hadamard(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales), M, N, K, group,
                                    int(hblock), _stream(stream)), "w4a16_gemv_hadamard")
    return (y, a) if a is not None else y


def selftest_wait_timeout(stream=None) -> None:
    """Launch the failure-path self-test: a kernel whose bounded wait cannot
    complete gives up and sets bit 2 of the device error word (device_error())."""
    _check(_lib.w4_selftest_wait_timeout(_stream(stream)), "w4_selftest_wait_timeout")


def _i32_scalar(t, name):
    _cuda(t, name)
    if t.dtype != torch.int32 or t.numel() < 1:
        raise ValueError(f"{name} must be a device int32 tensor")
    return t


def w4_kv_append(k_cache, v_cache, k_new, v_new, pos, kpos=None, status=None, stream=None):
    """Write k_new, v_new (bf16 [D]) into slot *pos mod T of a ring (kpos int32 [T]
    records *pos there) or slot *pos of a full cache (kpos None)."""
    _bits16(k_cache, "k_cache"); _bits16(v_cache, "v_cache"); _bits16(k_new, "k_new"); _bits16(v_new, "v_new")
    _i32_scalar(pos, "pos")
    T, D = k_cache.shape
    if tuple(v_cache.shape) != (T, D) or k_new.numel() != D or v_new.numel() != D:
        raise ValueError("cache / new-row shape mismatch")
    if kpos is not None and (kpos.dtype != torch.int32 or kpos.numel() != T):
        raise ValueError("kpos must be int32 [T]")
    _check(_lib.w4_kv_append(_ptr(k_cache), _ptr(v_cache), _ptr(kpos), _ptr(k_new), _ptr(v_new), _ptr(pos), T, D,
                             _ptr(status), _stream(stream)), "w4_kv_append")


def w4a16_gemv_argmax_forced(x, qweight, scales, forced, group: int = 32, out=None, argmax=None, stream=None):
    """Greedy LM head for one x-row; when the device int32 *forced >= 0 no weight is
    read, y is left unchanged and argmax[0] = *forced. Returns (y, argmax)."""
    _bits16(x, "x"); _u32(qweight, "qweight"); _bits16(scales, "scales")
    _i32_scalar(forced, "forced")
    M, N, K = _shape(x, qweight, scales, group)
    if M != 1:
        raise ValueError("the forced-token LM head takes one x-row")
    y = torch.empty((1, N), dtype=torch.float32, device=x.device) if out is None else _cuda(out, "out")
    a = torch.empty((1,), dtype=torch.int32, device=x.device) if argmax is None else _i32_scalar(argmax, "argmax")
    _check(_lib.w4a16_gemv_argmax_forced(_ptr(y), _ptr(a), _ptr(x), _ptr(qweight), _ptr(scales), N, K, group,
                                         _ptr(forced), _stream(stream)), "w4a16_gemv_argmax_forced")
    return y, a


def w4_decode_prologue(token, pos, qtable, scales, group: int = 32, x_next=None, tokens=None, status=None,
                       stream=None):
    """tok = *token; tokens[*pos + 1] = tok; *pos += 1; x_next = bf16 row tok of the
    4-bit table (as w4_embed_gather). Returns x_next (bf16 [1][K])."""
    _i32_scalar(token, "token"); _i32_scalar(pos, "pos"); _u32(qtable, "qtable"); _bits16(scales, "scales")
    V, K = qtable.shape[0], qtable.shape[1] * 8
    if tuple(scales.shape) != (V, K // group):
        raise ValueError("scales shape mismatch")
    cap = 0
    if tokens is not None:
        _i32_scalar(tokens, "tokens")
        cap = tokens.numel()
    o = torch.empty((1, K), dtype=torch.bfloat16, device=token.device) if x_next is None else _cuda(x_next, "x_next")
    _check(_lib.w4_decode_prologue(_ptr(o), _ptr(tokens), _ptr(pos), _ptr(token), _ptr(qtable), _ptr(scales), V, K,
                                   group, cap, _ptr(status), _stream(stream)), "w4_decode_prologue")
    return o
