"""The row-sharded multi-GPU split (one process per GPU, rows of each projection
split in whole 16-row blocks, x replicated, y and the greedy pick all-gathered)
on CPU: gloo ranks exchange slices that each rank computed with the oracle on
its own rows. The assembled y must be bitwise the unsharded oracle's and the
pick the unsharded oracle's index.

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch", the w4gemv paragraph
(decode multiplies one vector by every weight matrix: rows are independent).
"""
import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_row_range_partition():
    from bit_weight_only_w4a16_gb300.shard import row_range
    for N in (0, 1, 15, 16, 17, 1536, 2560, 262144, 262144 + 7, 33):
        for world in (1, 2, 3, 4, 8):
            ranges = [row_range(N, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == N
            for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
                assert a1 == b0  # contiguous, in rank order
            for r0, r1 in ranges:
                assert r0 % 16 == 0 and (r1 % 16 == 0 or r1 == N)  # whole row blocks
            blocks = [(r1 - r0 + 15) // 16 for r0, r1 in ranges]
            assert max(blocks) - min(blocks) <= 1  # balanced to one block


def test_combine_picks_rules():
    import torch
    from bit_weight_only_w4a16_gb300.shard import combine_picks
    vals = [torch.tensor([1.0, 5.0, -0.0, 2.0]), torch.tensor([3.0, 5.0, 0.0, 2.0]),
            torch.tensor([3.0, 4.0, 0.0, float("-inf")])]
    idxs = [torch.tensor([0, 10, 7, 40]), torch.tensor([20, 30, 3, 2]), torch.tensor([50, 60, 90, 100])]
    v, i = combine_picks(vals, idxs)
    # larger value wins; equal values: lower index; -0 == +0
    assert i.tolist() == [20, 10, 3, 2]
    assert v.tolist()[:2] == [3.0, 5.0]


def _rank_main(rank, world, port, out_path, cases):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import synth
    from bit_weight_only_w4a16_gb300 import shard
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = []
    try:
        for (seed, M, N, K, group) in cases:
            x = synth.gen_x(seed, M, K)
            qw = synth.gen_qweight(seed, N, K)
            sc = synth.gen_scales(seed, N, K, group)
            r0, r1 = shard.row_range(N, world, rank)
            if r1 > r0:
                yl, _ = oracle.gemm(x, qw[r0:r1], sc[r0:r1], group)
            else:
                yl = np.zeros((M, 0))
            yl_t = torch.from_numpy(np.ascontiguousarray(yl))
            y = shard.all_gather_rows(yl_t, N).numpy()
            # local greedy pick: lowest index of the largest local value
            if r1 > r0:
                li = yl.argmax(axis=1)
                val = torch.from_numpy(yl[np.arange(M), li].copy())
                gi = torch.from_numpy(li + r0)
            else:
                val = torch.full((M,), float("-inf"), dtype=torch.float64)
                gi = torch.full((M,), N, dtype=torch.int64)
            _, idx = shard.all_gather_picks(val, gi)
            yfull, afull = oracle.gemm(x, qw, sc, group)
            ok_y = bool(np.array_equal(y, yfull))
            want = [int(oracle.argmax(yfull[m])[0]) for m in range(M)]
            res.append({"case": [seed, M, N, K, group], "y_bitwise": ok_y, "idx": idx.tolist(), "want": want})
        with open(f"{out_path}.{rank}", "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_rows_and_pick_gloo(world):
    import torch.multiprocessing as mp
    cases = [(5000, 1, 2560, 1536, 32), (5001, 3, 1000, 512, 64), (5002, 2, 8193, 256, 128),
             (5003, 1, 40, 128, 32), (5004, 8, 4096, 384, 32)]
    port = _free_port()
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    out = os.path.join(out_dir, f"shard_{os.getpid()}_{world}")
    mp.spawn(_rank_main, args=(world, port, out, cases), nprocs=world, join=True)
    try:
        for r in range(world):
            with open(f"{out}.{r}") as f:
                res = json.load(f)
            for c in res:
                assert c["y_bitwise"], (r, c["case"])
                assert c["idx"] == c["want"], (r, c["case"], c["idx"], c["want"])
    finally:
        for r in range(world):
            if os.path.exists(f"{out}.{r}"):
                os.remove(f"{out}.{r}")
