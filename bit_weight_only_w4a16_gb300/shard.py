"""Row-sharded decode GEMV over several GPUs, one process per GPU.

Source: "Gemma 4 E2B on a 4 GB GPU with pure PyTorch" - the w4gemv paragraph:
decode multiplies one activation vector by every weight matrix, and each output
row depends on its own weight row only. So a projection splits across G GPUs by
rows: rank r holds a contiguous range of whole 16-row blocks of qweight and
scales (its slice of HBM traffic), x is replicated, the rank runs the library's
own decode kernels on its rows, and one all-gather assembles y (4 * M * N / G
bytes from each rank). The greedy pick over a sharded vocabulary gathers one
(largest logit, index) pair per x-row and rank and keeps the largest logit, the
lowest index among equal ones (-0 equal to +0), the same rule as the fused pick.

The pure helpers (row_range, assemble_rows, combine_picks) do no communication;
all_gather_rows and all_gather_picks exchange through torch.distributed (NCCL
between GPUs, gloo for host tensors) and need an initialised process group.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

ROW_BLOCK = 16  # rows of one decode row block; shards never split one


def row_range(N: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [r0, r1) of rank `rank`: whole 16-row blocks, split as evenly as
    possible (rank r gets blocks [nrb*r/world, nrb*(r+1)/world))."""
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError(f"bad shard request N={N} world={world} rank={rank}")
    nrb = (N + ROW_BLOCK - 1) // ROW_BLOCK
    b0, b1 = nrb * rank // world, nrb * (rank + 1) // world
    return min(N, ROW_BLOCK * b0), min(N, ROW_BLOCK * b1)


def assemble_rows(parts, N: int) -> torch.Tensor:
    """y [M][N] from the ranks' [M][r1 - r0] slices, in rank order."""
    world = len(parts)
    for r, p in enumerate(parts):
        r0, r1 = row_range(N, world, r)
        if p.shape[-1] != r1 - r0:
            raise ValueError(f"rank {r}: slice of {p.shape[-1]} rows, expected {r1 - r0}")
    return torch.cat(list(parts), dim=-1)


def _pick_better(v_new, i_new, v_best, i_best):
    """Mask of x-rows where (v_new, i_new) beats (v_best, i_best): a larger value,
    or an equal value (so -0 == +0) with a lower index."""
    return (v_new > v_best) | ((v_new == v_best) & (i_new < i_best))


def combine_picks(vals, idxs):
    """Global greedy pick per x-row from per-rank (value [M], global index [M])
    pairs. Returns (value [M], index [M]) of the winner."""
    if len(vals) != len(idxs) or not vals:
        raise ValueError("one (value, index) pair list per rank")
    bv, bi = vals[0].clone(), idxs[0].clone()
    for v, i in zip(vals[1:], idxs[1:]):
        take = _pick_better(v, i, bv, bi)
        bv = torch.where(take, v, bv)
        bi = torch.where(take, i, bi)
    return bv, bi


def all_gather_rows(y_local: torch.Tensor, N: int, group=None) -> torch.Tensor:
    """All-gather the ranks' row slices of y [M][n_local] into y [M][N]. Slices
    are padded to the widest one for the collective and trimmed after it."""
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    r0, r1 = row_range(N, world, rank)
    if y_local.shape[-1] != r1 - r0:
        raise ValueError(f"local slice has {y_local.shape[-1]} rows, expected {r1 - r0}")
    widths = [row_range(N, world, r)[1] - row_range(N, world, r)[0] for r in range(world)]
    wmax = max(widths)
    M = y_local.shape[0]
    send = torch.zeros((M, wmax), dtype=y_local.dtype, device=y_local.device)
    send[:, :r1 - r0] = y_local
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    return assemble_rows([recv[r][:, :widths[r]] for r in range(world)], N)


def all_gather_picks(val: torch.Tensor, idx: torch.Tensor, group=None):
    """All-gather each rank's (largest value, global index) per x-row and
    combine them (combine_picks). val fp32 [M], idx int [M]; the pair travels
    as exact fp64 so one collective carries both."""
    world = dist.get_world_size(group)
    pair = torch.stack([val.to(torch.float64), idx.to(torch.float64)], dim=0)
    recv = [torch.empty_like(pair) for _ in range(world)]
    dist.all_gather(recv, pair, group=group)
    v, i = combine_picks([p[0] for p in recv], [p[1].to(torch.int64) for p in recv])
    return v.to(val.dtype), i


def sharded_gemv(x, qweight_shard, scales_shard, N: int, group: int = 32, pg=None, stream=None):
    """y [M][N] of a row-sharded projection: this rank's rows with the library's
    decode kernels, then the all-gather. qweight_shard / scales_shard are the
    rank's rows row_range(N, world, rank) of the full tensors."""
    from . import w4a16_gemv
    if qweight_shard.shape[0] == 0:  # more ranks than row blocks: nothing here
        y_local = torch.empty((x.shape[0], 0), dtype=torch.float32, device=x.device)
    else:
        y_local = w4a16_gemv(x, qweight_shard, scales_shard, group=group, stream=stream)
    return all_gather_rows(y_local, N, pg)


def sharded_gemv_argmax(x, qweight_shard, scales_shard, N: int, group: int = 32, pg=None, stream=None):
    """(y [M][N], argmax [M]) of a row-sharded projection with the greedy pick:
    the local fused pick gives each rank's best (value, index); one all-gather
    of those pairs and one of the y slices."""
    from . import w4a16_gemv_argmax
    world, rank = dist.get_world_size(pg), dist.get_rank(pg)
    r0, _ = row_range(N, world, rank)
    M = x.shape[0]
    if qweight_shard.shape[0] == 0:  # more ranks than row blocks: no candidate here
        y_local = torch.empty((M, 0), dtype=torch.float32, device=x.device)
        val = torch.full((M,), float("-inf"), dtype=torch.float32, device=x.device)
        gidx = torch.full((M,), N, dtype=torch.int64, device=x.device)
    else:
        y_local, a_local = w4a16_gemv_argmax(x, qweight_shard, scales_shard, group=group, stream=stream)
        a64 = a_local.to(torch.int64)
        val = torch.gather(y_local, 1, a64[:, None])[:, 0]
        gidx = a64 + r0
    _, idx = all_gather_picks(val, gidx, pg)
    return all_gather_rows(y_local, N, pg), idx.to(torch.int32)
