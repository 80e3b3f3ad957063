"""The row-sharded split with the library's kernels computing each shard (GPU):
the shards' y assembled in rank order and the combined greedy pick against the
fp64 oracle, for 2, 3 and 4 shards run one after another on the one GPU, and
the NCCL all-gather path (world size 1) against the unsharded call."""
import os
import socket

import numpy as np
import pytest

import oracle
import synth
from _util import assert_w4_close, to_dev_bits16, to_dev_u32
from _guard import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import bit_weight_only_w4a16_gb300 as w4
    w4.init()
    return guarded(w4)


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("M,N,K,group", [(1, 20000, 1536, 32), (2, 4104, 2048, 64), (8, 3000, 1536, 256)])
def test_shards_assembled_match_oracle(w4, world, M, N, K, group):
    import torch
    from bit_weight_only_w4a16_gb300 import shard
    x, qw = synth.gen_x(5100 + M, M, K), synth.gen_qweight(5100 + N, N, K)
    sc = synth.gen_scales(5100 + N, N, K, group)
    xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
    parts, vals, idxs = [], [], []
    for r in range(world):
        r0, r1 = shard.row_range(N, world, r)
        y, a = w4.w4a16_gemv_argmax(xd, qd[r0:r1].contiguous(), sd[r0:r1].contiguous(), group=group)
        a64 = a.to(torch.int64)
        parts.append(y)
        vals.append(torch.gather(y, 1, a64[:, None])[:, 0])
        idxs.append(a64 + r0)
    y = shard.assemble_rows(parts, N).cpu().numpy()
    _, idx = shard.combine_picks(vals, idxs)
    yr, ar = oracle.gemm(x, qw, sc, group)
    assert_w4_close(y, yr, ar, what=f"{world} shards")
    for m in range(M):
        want, gap = oracle.argmax(yr[m])
        assert gap > 2 * (1e-4 * ar[m, want] + 1e-6), "ambiguous seed"
        assert int(idx[m]) == want


def test_nccl_all_gather_path_world1(w4):
    import torch
    import torch.distributed as dist
    from bit_weight_only_w4a16_gb300 import shard
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        M, N, K = 2, 9000, 1536
        x, qw, sc = synth.gen_w4_problem(5200, M, N, K)
        xd, qd, sd = to_dev_bits16(x), to_dev_u32(qw), to_dev_bits16(sc)
        y, idx = shard.sharded_gemv_argmax(xd, qd, sd, N)
        y2 = shard.sharded_gemv(xd, qd, sd, N)
        yp, ap = w4.w4a16_gemv_argmax(xd, qd, sd)
        torch.cuda.synchronize()
        assert torch.equal(y, yp) and torch.equal(y2, yp)
        assert torch.equal(idx, ap)
    finally:
        dist.destroy_process_group()
