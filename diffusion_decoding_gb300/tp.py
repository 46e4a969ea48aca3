"""Tensor-parallel vocabulary sharding of the decode statistics (plumbing only).

With the output layer split over the tensor-parallel group (dInfer explainer, system
optimisations), rank k holds the logits of one contiguous vocabulary range.  Each rank reduces
its own columns with ``dllm_decode_stats``; the exchange step gathers every rank's per-row
(row_max, lse, argmax) from all ranks with ``torch.distributed.all_gather``; then each rank merges
them with ``dllm_merge_shard_stats`` (a CUDA kernel) and holds identical whole-vocabulary
statistics, from which it runs the same commit (``logits=None``).  Only argument marshalling and
the collective live here: every step of the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def vocab_range(V: int, world: int, rank: int) -> tuple[int, int]:
    """(first id, count) of rank's contiguous share of V ids; shares differ by at most one."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a group of {world}")
    base, extra = divmod(V, world)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def all_gather_shard_stats(stats, group=None):
    """Gather every rank's (row_max, lse, argmax) of the same rows.

    stats: any object with row_max, lse (float32) and argmax (int32) tensors of R rows on this
    rank's device (e.g. ``StatsBuffers``).  Returns a list, one entry per rank in rank order, of
    objects with the same three fields plus a fresh ``conf`` tensor (unused by the merge)."""
    world = dist.get_world_size(group)
    fields = ("row_max", "lse", "argmax")
    gathered = {f: [torch.empty_like(getattr(stats, f)) for _ in range(world)] for f in fields}
    for f in fields:
        dist.all_gather(gathered[f], getattr(stats, f).contiguous(), group=group)
    out = []
    for k in range(world):
        g = type("ShardStats", (), {})()
        for f in fields:
            setattr(g, f, gathered[f][k])
        g.conf = torch.empty_like(gathered["lse"][k])
        out.append(g)
    return out


def merge_gathered(gathered, V: int, out, stream=None) -> None:
    """Merge the gathered shard statistics (rank order) into ``out`` on this rank's GPU."""
    import diffusion_decoding_gb300 as dd
    world = len(gathered)
    shards = [(g, vocab_range(V, world, k)[0]) for k, g in enumerate(gathered)]
    dd.dllm_merge_shard_stats(shards, gathered[0].row_max.numel(), out, stream)
