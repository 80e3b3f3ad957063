"""The decode weight sweep exactly as the benchmark times it: all 140 fused
calls of the 35-layer model (1.02 GB of packed weights) captured in one CUDA
graph with programmatic dependent launch and replayed, at M = 1 and M = 8.
Sampled rows of every stage shape (first and last layer) are checked against
the fp64 oracle with the decode bar |y - y_ref| <= 1e-4 * sum|w x| + 1e-6.

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph
(one vector times every weight matrix per token) and the CUDA-graph paragraph
(the step captured once and replayed).
"""
import numpy as np
import pytest

import bench
import oracle
import synth
from _util import assert_w4_close
from _guard import Guard

pytestmark = pytest.mark.gpu


def _stage_rows(stage, rows):
    """Host codes and steps of the given rows of a fused stage (the members'
    generators, as the benchmark's arena was filled)."""
    l, K = stage["layer"], stage["K"]
    members = next(m for nm, m, _, _ in bench.fused_stages(l) if nm == stage["name"])
    qs, ss, r0 = [], [], 0
    for p in members:
        n_p = next(n for nm, n, _ in bench.layer_shapes(l) if nm == p)
        sel = rows[(rows >= r0) & (rows < r0 + n_p)] - r0
        if sel.size:
            qs.append(synth.gen_qweight(bench.seed_of(l, p), n_p, K)[sel])
            ss.append(synth.gen_scales(bench.seed_of(l, p), n_p, K)[sel])
        r0 += n_p
    return np.concatenate(qs), np.concatenate(ss)


@pytest.mark.parametrize("M", [1, 8])
def test_graph_replayed_sweep_sampled_rows(M):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    dev = torch.device("cuda", 0)
    sweep = bench.Sweep(dev, keep_host=False, m=M)
    # Each stage's y inside guard bands: a write past one stage's output would
    # otherwise land unseen in the next stage's.
    guards = []
    for st in sweep.stages:
        g = Guard((M, st["N"]), torch.float32, device=dev)
        st["y"] = g.t
        guards.append(g)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sweep.run(w4, stream)
    torch.cuda.synchronize()
    for st in sweep.stages:
        st["y"].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep.run(w4, stream)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert w4.device_error() == 0
    for i, g in enumerate(guards):
        g.check(f"sweep M={M} stage {i}")
    n = len(sweep.stages)
    picks = list(range(4)) + list(range(n - 4, n))  # every fused shape, layers 0 and 34
    rng = np.random.default_rng(1234 + M)
    for i in picks:
        st = sweep.stages[i]
        N, K = st["N"], st["K"]
        rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 46, replace=False)]))
        qw, sc = _stage_rows(st, rows)
        x = synth.gen_x(bench.seed_of(st["layer"], next(m for nm, m, _, _ in bench.fused_stages(st["layer"])
                                                        if nm == st["name"])[0]), M, K)
        yr, ar = oracle.gemm(x, qw, sc, 32)
        y = st["y"].cpu().numpy()[:, rows]
        assert np.isfinite(y).all()
        assert_w4_close(y, yr, ar, what=f"sweep M={M} stage {i} ({st['name']} {N}x{K})")
