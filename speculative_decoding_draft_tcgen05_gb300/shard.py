"""Host side of the vocabulary-sharded selector: which lm_head rows each rank
holds, and the exchange of the ranks' top-K lists.

The K best tokens of a position over the whole vocabulary are the K best of
the union of every shard's K best (blog "DFlash 2: Keep Drafting Parallel",
"A Lightweight Path Selector": the selector keeps the drafter's K best
candidates of each position). Each rank streams its rows of the lm_head with
``dflash_select_topk_shard``, the [B, L, K] lists are all-gathered into
[G, B, L, K], and every rank finishes with ``dflash_select_run_gathered``.
The exchange moves G * B * L * K * 8 bytes per step (7 KB per rank at batch 1,
L = 7, K = 16).
"""
from __future__ import annotations


def shard_range(V: int, G: int, rank: int) -> tuple[int, int]:
    """Rows [v0, v1) of rank ``rank`` out of G: contiguous, disjoint, covering
    [0, V), whole 128-row tiles except the last shard's tail, sizes differing
    by at most one tile."""
    if not 0 <= rank < G or V < 1:
        raise ValueError(f"rank {rank} of {G} over {V} rows")
    tiles = (V + 127) // 128
    base, extra = divmod(tiles, G)
    t0 = rank * base + min(rank, extra)
    t1 = t0 + base + (1 if rank < extra else 0)
    return min(V, 128 * t0), min(V, 128 * t1)


def all_gather_keys(keys, group=None):
    """All-gathers every rank's [B, L, K] key list (int64 tensor, on the
    device with NCCL or on the host with gloo) into [G, B, L, K], rank order."""
    import torch
    import torch.distributed as dist
    G = dist.get_world_size(group)
    keys = keys.contiguous()
    out = torch.empty((G * keys.shape[0],) + tuple(keys.shape[1:]), dtype=keys.dtype, device=keys.device)
    dist.all_gather_into_tensor(out, keys, group=group)  # concatenated along dim 0, rank order
    return out.view((G,) + tuple(keys.shape))
