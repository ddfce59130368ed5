"""Context-parallel prefill: the sequence split over ranks and the one
all-gather that gives every rank the whole sequence's cache entries.

DSA page, "并行：为什么 DSA 偏爱 CP": the indexer sums over heads before its
top-k, so it cannot be split by head; split by sequence instead.  Each rank
keeps its own share of the queries, builds the cache entries of its own
tokens, and one all-gather (no ring) brings every rank the entries of the
whole sequence, reordered to sequence order; the indexer, top-k and sparse
attention then run locally with no further exchange.  An all-gather wants the
same shape on every rank, so each rank pads its share to the largest share
and the receiver drops the padding.

Two ways to balance the causal work ("怎么切 Q：zigzag 与 interleave"):
  * interleave: unit u goes to rank u % p;
  * zigzag: the units are cut into 2p consecutive blocks, and rank r takes
    blocks r and 2p - 1 - r (a head block paired with a tail block).
Reading for CSA2: the unit is a cache entry (m consecutive tokens, m = 1 or
2), not a token, because an entry's compression pools the m tokens of that
entry and they must be on one rank; a rank's queries are the tokens of its
entries.

The exchange runs through torch.distributed (NCCL between GPUs, gloo in the
CPU tests); the reorder is a row scatter.  The entries themselves are built
by csa2_compress_m2 on each rank before the gather.
"""
from __future__ import annotations

import torch

STRATEGIES = ("interleave", "zigzag")


def cp_units(n_units: int, world: int, rank: int, strategy: str = "interleave") -> torch.Tensor:
    """Ascending ids (int64) of the units (cache entries) owned by `rank`."""
    if strategy not in STRATEGIES:
        raise ValueError(f"strategy {strategy!r} is not one of {STRATEGIES}")
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} not in 0..{world - 1}")
    if strategy == "interleave":
        return torch.arange(rank, max(rank, n_units), world, dtype=torch.int64)
    nb = 2 * world
    cut = [b * n_units // nb for b in range(nb + 1)]
    lo, hi = rank, nb - 1 - rank
    return torch.cat([torch.arange(cut[lo], cut[lo + 1], dtype=torch.int64),
                      torch.arange(cut[hi], cut[hi + 1], dtype=torch.int64)])


def cp_tokens(n_units: int, ratio_m: int, world: int, rank: int, strategy: str = "interleave") -> torch.Tensor:
    """Token positions (the rank's query rows) of the rank's units: m per unit."""
    u = cp_units(n_units, world, rank, strategy)
    return (u[:, None] * ratio_m + torch.arange(ratio_m, dtype=torch.int64)[None, :]).reshape(-1)


def cp_causal_pairs(n_units: int, ratio_m: int, world: int, rank: int, strategy: str = "interleave") -> int:
    """Query-entry pairs the rank's indexer scores under the causal mask: a
    query at position i sees the entries (i + 1) // m."""
    t = cp_tokens(n_units, ratio_m, world, rank, strategy)
    return int(((t + 1) // ratio_m).sum())


def cp_all_gather(local: torch.Tensor, n_units: int, world: int, rank: int, strategy: str = "interleave",
                  group=None) -> torch.Tensor:
    """All ranks' unit rows in unit order.  `local` holds this rank's rows
    [len(cp_units(...)), ...] in ascending unit order; returns [n_units, ...]."""
    import torch.distributed as dist
    mine = cp_units(n_units, world, rank, strategy)
    if local.shape[0] != mine.numel():
        raise ValueError(f"rank {rank} holds {local.shape[0]} rows, its share is {mine.numel()}")
    shares = [cp_units(n_units, world, r, strategy) for r in range(world)]
    width = max(s.numel() for s in shares)
    padded = local.new_zeros((width,) + tuple(local.shape[1:]))
    padded[:local.shape[0]] = local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded, group=group)
    out = local.new_empty((n_units,) + tuple(local.shape[1:]))
    for r, ids in enumerate(shares):
        out.index_copy_(0, ids.to(out.device), parts[r][:ids.numel()])
    return out


def cp_gather_bytes_per_rank(n_units: int, unit_bytes: int, world: int, strategy: str = "interleave") -> int:
    """Bytes a rank receives in the all-gather: the p - 1 other ranks' padded
    shares of unit_bytes each, about (p - 1) / p * n_units * unit_bytes (the
    O(S) volume of the DSA page's comparison table)."""
    width = max(cp_units(n_units, world, r, strategy).numel() for r in range(world))
    return (world - 1) * width * unit_bytes
