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


def attn_rel_bound(D, S, T):
    """Relative bound of the decode attention (times sum_t w_t |v_t|), derived
    from the kernel's arithmetic:
      2^-16            the value product applies hi + lo of each weight (two bf16
                       parts, within 2^-18 of the kernel's fp32 weight) and the
                       normaliser adds those applied weights: a convex combination
                       with weights within 2 * 2^-18 relative, doubled for margin;
      2^-19            exp2f (2 ulp) and the roundings of its argument;
      2 D 2^-23 S      the fp32 score sums over D products (S = max over kept
                       slots of scale * sum_d |q_d k_d|; a score error e moves a
                       weight by at most a factor e^(2e));
      (2 T/16 + 64) 2^-23  the fp32 accumulation of the outputs and the normaliser
                       along the longest chain: a rescale and an add per 16-token
                       tile (all tiles in one slice at worst), the mma's own sums
                       and the merge of the slices."""
    import math
    return 2.0 ** -16 + 2.0 ** -19 + 2.0 * D * 2.0 ** -23 * S + (2 * math.ceil(T / 16) + 64) * 2.0 ** -23
