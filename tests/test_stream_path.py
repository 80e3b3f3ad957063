"""The bulk-copy streaming decode kernel (gemv_stream.cu) is not chosen by the
per-shape table on GB300 (the register kernel measured faster on every sweep
shape), so these tests force it with W4_DECODE_PATH=stream in a child process
(the library reads the variable once) and check it against the oracle."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import bit_weight_only_w4a16_gb300 as w4
import synth, oracle
from tests._util import assert_w4_close, to_dev_bits16, to_dev_u32
torch.cuda.set_device(0)
for (M, N, K, seed) in [(1, 2560, 1536, 81), (2, 1536, 6144, 82), (1, 500, 2048, 83), (2, 300, 12288, 84)]:
    x, qw, sc = synth.gen_w4_problem(seed, M, N, K)
    y = w4.w4a16_gemv(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc))
    yr, ar = oracle.gemm(x, qw, sc)
    assert_w4_close(y.cpu().numpy(), yr, ar, what=f"stream {{M}}x{{N}}x{{K}}")
    ya, a = w4.w4a16_gemv_argmax(to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc))
    torch.cuda.synchronize()
    assert np.array_equal(ya.cpu().numpy().view(np.uint32), y.cpu().numpy().view(np.uint32))
    for m in range(M):
        assert int(a[m]) == int(np.flatnonzero(ya[m].cpu().numpy() == ya[m].max().item())[0])
assert w4.device_error() == 0
print("ok")
"""


@pytest.mark.gpu
def test_forced_stream_kernel_matches_oracle():
    env = dict(os.environ, W4_DECODE_PATH="stream")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
