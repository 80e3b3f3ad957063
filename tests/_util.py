"""Helpers shared by the tests: device transfer of generator output and the tolerance rule."""
import numpy as np


def torch_dev():
    import torch
    return torch.device("cuda", torch.cuda.current_device())


def to_dev_u32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(torch_dev())


def to_dev_bits16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(torch_dev())


def bits16(t):
    """Raw uint16 bits of a device bf16/int16 tensor."""
    import torch
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy().view(np.uint16)


def assert_w4_close(y, y_ref, absy, rel=1e-4, abs_=1e-6, what=""):
    """|y - y_ref| <= rel * sum|w x| + abs_, elementwise (the GEMV parity bar)."""
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - y_ref)
    bound = rel * absy + abs_
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={y_ref[tuple(i)]!r} err={err[tuple(i)]:.3e} "
                             f"bound={bound[tuple(i)]:.3e}")
    return float((err / np.maximum(absy, 1e-30)).max())
