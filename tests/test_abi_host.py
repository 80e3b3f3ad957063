"""Host-side checks of the C ABI: the library builds, loads, exports every symbol
the header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import bit_weight_only_w4a16_gb300 as w4
    path = w4.LIB_PATH
    return w4._lib, path


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("w4a16_gemv", "w4a16_gemm", "w4a16_gemv_argmax", "w4_embed_gather", "hbm_read_probe",
              "w4_init", "w4_status_string", "w4_last_cuda_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    l, path = lib
    for n in _declared():
        assert hasattr(l, n), n
    import bit_weight_only_w4a16_gb300 as w4
    assert set(w4.EXPORTS) <= set(_declared())


def test_status_strings(lib):
    l, _ = lib
    assert l.w4_status_string(0) == b"W4_OK"
    assert l.w4_status_string(3) == b"W4_ERR_MISALIGNED"
    assert l.w4_status_string(99) == b"W4_ERR_UNKNOWN"


def _addr(v):
    return ctypes.c_void_p(v)


def test_validation_before_any_launch(lib):
    import torch
    if torch.cuda.is_available():
        # Fake addresses: never handed to a machine where a launch could use them.
        pytest.skip("host-only check (a GPU is present)")
    l, _ = lib
    A = _addr(1 << 20)  # a 16-byte aligned non-NULL address; never dereferenced
    # NULL pointer
    assert l.w4a16_gemv(None, A, A, A, 1, 16, 64, 32, None) == 1
    # sizes
    assert l.w4a16_gemv(A, A, A, A, 0, 16, 64, 32, None) == 1
    assert l.w4a16_gemv(A, A, A, A, 1, -1, 64, 32, None) == 1
    assert l.w4a16_gemv(A, A, A, A, 1, 16, 48, 32, None) == 1
    # group outside {32, 64, 128, 256, 512}
    assert l.w4a16_gemv(A, A, A, A, 1, 16, 96, 48, None) == 2
    assert l.w4a16_gemv(A, A, A, A, 1, 16, 1024, 1024, None) == 2
    assert l.w4a16_gemv(A, A, A, A, 1, 16, 64, 16, None) == 2
    assert l.w4_embed_gather(A, A, A, A, 1, 10, 96, 48, None, None) == 2
    # K not a multiple of a served group
    assert l.w4a16_gemv(A, A, A, A, 1, 16, 96, 64, None) == 1
    # M beyond the decode call
    assert l.w4a16_gemv(A, A, A, A, 9, 16, 64, 32, None) == 2
    assert l.w4a16_gemv_argmax(A, A, A, A, A, 9, 16, 64, 32, None) == 2
    # misaligned
    assert l.w4a16_gemv(A, _addr((1 << 20) + 2), A, A, 1, 16, 64, 32, None) == 3
    assert l.w4a16_gemv(A, A, _addr((1 << 20) + 4), A, 1, 16, 64, 32, None) == 3
    # index overflow
    assert l.w4a16_gemv(A, A, A, A, 1, 1 << 30, 64, 32, None) == 1
    # gather / probe
    assert l.w4_embed_gather(A, A, A, A, 1, 10, 40, 32, None, None) == 1
    assert l.w4_embed_gather(A, None, A, A, 1, 10, 64, 32, None, None) == 1
    assert l.hbm_read_probe(A, A, ctypes.c_size_t(24), None) == 1
    assert l.hbm_read_probe(A, _addr((1 << 20) + 8), ctypes.c_size_t(32), None) == 3
    # prefill shape rules
    assert l.w4a16_gemm(A, A, A, A, 64, 24, 64, 32, None) == 2
    assert l.w4a16_gemm(A, A, A, A, 64, 32, 96, 32, None) == 2
    # Hadamard-rotated GEMV: block size, K multiple, rows
    assert l.w4a16_gemv_hadamard(A, None, A, A, A, 1, 16, 1024, 32, 96, None) == 2
    assert l.w4a16_gemv_hadamard(A, None, A, A, A, 1, 16, 1024, 32, 8192, None) == 2
    assert l.w4a16_gemv_hadamard(A, None, A, A, A, 1, 16, 1024, 32, 2048, None) == 1
    assert l.w4a16_gemv_hadamard(A, None, A, A, A, 5, 16, 1024, 32, 256, None) == 2
    assert l.w4a16_gemv_hadamard(A, _addr((1 << 20) + 2), A, A, A, 1, 16, 1024, 32, 256, None) == 3
    # decode attention: NULL, sizes, head count / width, alignment
    f = ctypes.c_float(1.0)
    assert l.w4_attn_decode(None, A, A, A, None, 0, 0, 8, 16, 512, f, None) == 1
    assert l.w4_attn_decode(A, A, A, A, None, 0, 0, 8, 0, 512, f, None) == 1
    assert l.w4_attn_decode(A, A, A, A, None, 0, -1, 8, 16, 512, f, None) == 1
    assert l.w4_attn_decode(A, A, A, A, None, 0, 0, 9, 16, 512, f, None) == 2
    assert l.w4_attn_decode(A, A, A, A, None, 0, 0, 8, 16, 200, f, None) == 2
    assert l.w4_attn_decode(A, A, A, A, None, 0, 0, 8, 16, 1024, f, None) == 2
    assert l.w4_attn_decode(A, A, _addr((1 << 20) + 8), A, None, 0, 0, 8, 16, 512, f, None) == 3
    assert l.w4_attn_decode(A, A, A, A, _addr((1 << 20) + 2), 0, 0, 8, 16, 512, f, None) == 3
    assert l.w4_attn_decode(A, A, A, A, None, 0, 0, 8, 1 << 22, 512, f, None) == 1
    # attention at a device position: the same checks plus the position pointer
    assert l.w4_attn_decode_devpos(A, A, A, A, None, None, 0, 8, 16, 512, f, None) == 1
    assert l.w4_attn_decode_devpos(A, A, A, A, None, A, 0, 9, 16, 512, f, None) == 2
    assert l.w4_attn_decode_devpos(A, A, A, A, None, _addr((1 << 20) + 2), 0, 8, 16, 512, f, None) == 3
    # key/value append: NULL, width, alignment
    assert l.w4_kv_append(A, A, None, A, A, None, 16, 512, None, None) == 1
    assert l.w4_kv_append(A, A, None, A, A, A, 16, 100, None, None) == 1
    assert l.w4_kv_append(A, A, None, A, A, A, 0, 512, None, None) == 1
    assert l.w4_kv_append(A, A, None, _addr((1 << 20) + 8), A, A, 16, 512, None, None) == 3
    assert l.w4_kv_append(A, A, _addr((1 << 20) + 2), A, A, A, 16, 512, None, None) == 3
    # forced-token LM head: NULL forced, group, alignment
    assert l.w4a16_gemv_argmax_forced(A, A, A, A, A, 16, 64, 32, None, None) == 1
    assert l.w4a16_gemv_argmax_forced(A, None, A, A, A, 16, 64, 32, A, None) == 1
    assert l.w4a16_gemv_argmax_forced(A, A, A, A, A, 16, 96, 48, A, None) == 2
    assert l.w4a16_gemv_argmax_forced(A, A, A, A, A, 16, 64, 32, _addr((1 << 20) + 2), None) == 3
    # prologue: NULL, sizes, group, history capacity, alignment
    assert l.w4_decode_prologue(A, None, A, None, A, A, 16, 64, 32, 0, None, None) == 1
    assert l.w4_decode_prologue(A, None, A, A, A, A, 0, 64, 32, 0, None, None) == 1
    assert l.w4_decode_prologue(A, A, A, A, A, A, 16, 64, 32, 0, None, None) == 1
    assert l.w4_decode_prologue(A, None, A, A, A, A, 16, 96, 48, 0, None, None) == 2
    assert l.w4_decode_prologue(A, None, A, A, A, A, 16, 96, 64, 0, None, None) == 1
    assert l.w4_decode_prologue(_addr((1 << 20) + 8), None, A, A, A, A, 16, 64, 32, 0, None, None) == 3


def test_no_device_reported_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    l, _ = lib
    assert l.w4_init() == 5
