"""Row sharding of one weight matrix across ranks (one process per GPU).

Output rows of Y = X . deq(W)^T are independent: row n of W produces column n
of Y and nothing else.  So the natural data-parallel split gives each rank a
contiguous range of weight rows (packed on that rank only), replicates the
activations, and concatenates the per-rank Y column ranges -- with no
exchange at all if the consumer takes sharded Y, or one all-gather otherwise.
Ranges are multiples of 16 rows (the kernels' row tile) except the last.
"""
from __future__ import annotations

ROW_ALIGN = 16


def row_shard(N: int, world: int, rank: int, align: int = ROW_ALIGN) -> tuple[int, int]:
    """[start, stop) weight rows owned by `rank` of `world` (balanced, aligned)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    tiles = (N + align - 1) // align
    lo = (tiles * rank) // world
    hi = (tiles * (rank + 1)) // world
    return min(lo * align, N), min(hi * align, N)


def shard_inputs(codes_canonical, scales_fp16, N: int, world: int, rank: int):
    """This rank's rows of the canonical codes and scales (host arrays)."""
    start, stop = row_shard(N, world, rank)
    return codes_canonical[start:stop], scales_fp16[start:stop], start, stop


def gather_columns(y_shard, N: int, group=None):
    """All-gather per-rank Y[T, rows of rank] into the full Y[T, N] (torch tensors).

    Uses torch.distributed (NCCL for GPU tensors, gloo for CPU tensors); the
    shards may differ in width, so they are padded to the widest before the
    collective and trimmed after it.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    T = y_shard.shape[0]
    widths = [row_shard(N, world, r)[1] - row_shard(N, world, r)[0] for r in range(world)]
    wmax = max(widths)
    padded = torch.zeros((T, wmax), dtype=y_shard.dtype, device=y_shard.device)
    padded[:, : y_shard.shape[1]] = y_shard
    bufs = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(bufs, padded, group=group)
    return torch.cat([b[:, :w] for b, w in zip(bufs, widths)], dim=1)
