"""Guard bands around every device output of the library, for the GPU tests.

A memory checker (compute-sanitizer) is not available for these tests, and an
elementwise comparison of an output cannot see a write past its end or before
its start. So every output buffer a test hands to the library sits inside a
larger allocation whose first and last 4 KiB (plus the rounding tail) hold a
fixed NaN bit pattern that no kernel of the library writes; after the call has
finished the bands must be bitwise unchanged.

`guarded(w4)` wraps the binding module: every call allocates the outputs it
would have allocated itself inside such bands, synchronises the device (unless
the current stream is capturing a CUDA graph) and checks the bands of those
outputs and of any guarded tensor passed in (caches, histories, position words
that the call updates in place). `Guard(shape, dtype)` makes a guarded tensor
for the tests that pass their own buffers.
"""
import weakref

import numpy as np

PAD = 4096                 # bytes of guard band on each side
PATTERN = 0x7FBADBAD       # an fp32 NaN payload (also not a plausible index or bf16 pair)

_live = {}                 # data_ptr of a guarded tensor -> weak reference to its Guard


def _torch():
    import torch
    return torch


class Guard:
    """A device tensor of `shape`/`dtype` surrounded by guard bands."""

    def __init__(self, shape, dtype, device=None, init=None):
        torch = _torch()
        if isinstance(shape, int):
            shape = (shape,)
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        body = (self.nbytes + 255) // 256 * 256
        self.raw = torch.empty(PAD + body + PAD, dtype=torch.uint8, device=dev)
        self.raw.view(torch.int32).fill_(PATTERN - (1 << 32) if PATTERN >= 1 << 31 else PATTERN)
        self.ref = self.raw.clone()
        self.t = self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)
        self.t._w4_guard = self    # the tensor keeps its guard (and bands) alive
        _live[self.t.data_ptr()] = weakref.ref(self)

    def bands_ok(self):
        lo = slice(0, PAD)
        hi = slice(PAD + self.nbytes, self.raw.numel())
        return bool(_torch().equal(self.raw[lo], self.ref[lo]) and _torch().equal(self.raw[hi], self.ref[hi]))

    def check(self, what=""):
        if not self.bands_ok():
            torch = _torch()
            lo = (self.raw[:PAD] != self.ref[:PAD]).nonzero()
            hi = (self.raw[PAD + self.nbytes:] != self.ref[PAD + self.nbytes:]).nonzero()
            raise AssertionError(f"{what}: write outside the output buffer "
                                 f"({lo.numel()} bytes changed before it, {hi.numel()} after it; "
                                 f"first before at {lo[0].item() - PAD if lo.numel() else None}, "
                                 f"first after at +{hi[0].item() if hi.numel() else None})")


def guard_of(t):
    torch = _torch()
    if isinstance(t, torch.Tensor) and t.is_cuda:
        g = getattr(t, "_w4_guard", None)
        if g is not None:
            return g
        r = _live.get(t.data_ptr())
        return r() if r is not None else None
    return None


def check_all(what=""):
    """Check every guard still alive (after a graph replay, say)."""
    _torch().cuda.synchronize()
    for r in list(_live.values()):
        g = r()
        if g is not None:
            g.check(what)


def forget_all():
    _live.clear()


def _gemv_out(a, kw):
    x, qw = a[0], a[1]
    return {"out": ((x.shape[0], qw.shape[0]), "float32")}


def _argmax_out(a, kw):
    d = _gemv_out(a, kw)
    d["argmax"] = ((a[0].shape[0],), "int32")
    return d


def _forced_out(a, kw):
    return {"out": ((1, a[1].shape[0]), "float32"), "argmax": ((1,), "int32")}


def _hadamard_out(a, kw):
    d = _gemv_out(a, kw)
    if kw.get("argmax") is True:
        d["argmax"] = ((a[0].shape[0],), "int32")
    return d


def _gather_out(a, kw):
    ids, qt = a[0], a[1]
    return {"out": ((ids.numel(), qt.shape[1] * 8), "bfloat16")}


def _attn_out(a, kw):
    q = a[0]
    return {"out": ((q.shape[0], q.shape[1]), "float32")}


def _probe_out(a, kw):
    return {"out": ((1,), "int64")}


def _prologue_out(a, kw):
    return {"x_next": ((1, a[2].shape[1] * 8), "bfloat16")}


# Outputs each call allocates when the caller passes none: name -> (shape, dtype).
_OUTPUTS = {
    "w4a16_gemv": _gemv_out,
    "w4a16_gemm": _gemv_out,
    "w4a16_gemv_argmax": _argmax_out,
    "w4a16_gemv_argmax_noalloc": _argmax_out,
    "w4a16_gemv_argmax_forced": _forced_out,
    "w4a16_gemv_hadamard": _hadamard_out,
    "w4_embed_gather": _gather_out,
    "w4_attn_decode": _attn_out,
    "hbm_read_probe": _probe_out,
    "w4_decode_prologue": _prologue_out,
    "w4_kv_append": lambda a, kw: {},
}


class _Guarded:
    def __init__(self, mod):
        self._mod = mod

    def __getattr__(self, name):
        f = getattr(self._mod, name)
        spec = _OUTPUTS.get(name)
        if spec is None:
            return f
        torch = _torch()

        def call(*args, **kw):
            mine = []
            for pname, (shape, dt) in spec(args, kw).items():
                v = kw.get(pname)
                if v is None or v is True:
                    g = Guard(shape, getattr(torch, dt), device=args[0].device)
                    kw[pname] = g.t
                    mine.append(g)
            passed = [g for g in (guard_of(v) for v in list(args) + list(kw.values())) if g is not None]
            r = f(*args, **kw)
            if not torch.cuda.is_current_stream_capturing():
                torch.cuda.synchronize()
                for g in mine + passed:
                    g.check(name)
            return r

        return call


def guarded(mod):
    """The binding module with guard bands around every output (see module doc)."""
    return _Guarded(mod)


def gzeros(shape, dtype, device=None):
    g = Guard(shape, dtype, device)
    g.t.zero_()
    return g.t


def gfull(shape, value, dtype, device=None):
    g = Guard(shape, dtype, device)
    g.t.fill_(value)
    return g.t


def gempty(shape, dtype, device=None):
    return Guard(shape, dtype, device).t


def gfrom(array, device=None):
    """A guarded device copy of a numpy array."""
    torch = _torch()
    src = torch.from_numpy(np.ascontiguousarray(array))
    g = Guard(tuple(src.shape), src.dtype, device)
    g.t.copy_(src)
    return g.t
