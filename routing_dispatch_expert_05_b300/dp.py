"""Data parallelism over token shards with a capacity over the whole batch.

Without a capacity limit a token's output depends on that token alone, and
R ranks run R independent replicas with no exchange.  A capacity factor
changes that.  "Expert Networks > Code Implementation" (In[10]) defines the
capacity over the batch as int(cf * (N // E)) and drops assignments in token
order, so whether a rank may keep an assignment depends on how many
assignments to the same expert the tokens before it made, on other ranks.

Rank r holds the r-th contiguous shard of the batch's N tokens (n_r tokens;
shards may differ in size).  The exchange step is:

  1. each rank routes its tokens and counts its selections per expert,
     before any drop (counts_r[e]);
  2. one all-gather of those E counts and n_r from every rank;
  3. prior_r[e] = sum over q < r of counts_q[e] (an exclusive scan over
     ranks);
  4. rank r keeps an assignment to e while its arrival index among the
     rank's own assignments to e is below room_r[e] = clamp(cap - prior_r[e],
     0, cap).  That is exactly the set the token-order rule keeps on the
     whole batch: an assignment's index in the batch is prior_r[e] plus its
     index in the shard.

The balance statistic ("Tutorial -- MoE SER Expert Routing", section 4) is
taken over the whole batch.  One all-reduce of the E selection counts and
the E per-expert probability sums gives
B = coef * sum_e (C_e / N) * (P_e / N) on every rank, and kept and dropped
add over ranks.

This module is the host side: the capacities (integer arithmetic) and the
orchestration over torch.distributed.  The per-rank stages are passed in as
callables.  The library's grouping entry point takes one capacity for all
experts, so on a GPU the per-expert room needs a grouping call that takes
an [E] array; with no capacity the ranks are plain replicas.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np


def global_capacity(capacity_factor: float, n_tokens_global: int, n_experts: int) -> Optional[int]:
    """int(cf * (N // E)) over the whole batch; None when cf <= 0 (no limit)."""
    if capacity_factor is None or capacity_factor <= 0:
        return None
    return int(capacity_factor * (n_tokens_global // n_experts))


def prior_counts(counts_all: np.ndarray, rank: int) -> np.ndarray:
    """Selections per expert made by the ranks before `rank` (exclusive scan
    over ranks of the all-gathered [R, E] counts)."""
    counts_all = np.asarray(counts_all, np.int64)
    return counts_all[:rank].sum(axis=0)


def shard_room(counts_all: np.ndarray, rank: int, capacity: Optional[int]) -> Optional[np.ndarray]:
    """How many assignments to each expert rank `rank` may keep."""
    if capacity is None:
        return None
    return np.clip(capacity - prior_counts(counts_all, rank), 0, capacity)


def balance_statistic(counts_total, psum_total, n_tokens_global: int, coef: float) -> float:
    """coef * sum_e (C_e / N) * (P_e / N) from the batch's totals."""
    c = np.asarray(counts_total, np.float64)
    p = np.asarray(psum_total, np.float64)
    n = float(n_tokens_global)
    return float(coef * np.sum((c / n) * (p / n)))


def dp_forward(x, route: Callable, dispatch: Callable, experts: Callable, combine: Callable,
               n_experts: int, capacity_factor: float, coef: float, group=None):
    """The layer forward for this rank's contiguous shard x of the batch.

    route(x) -> (idx [n, k], w [n, k], p [n, E]); dispatch(idx, x, room) ->
    (offsets, row_of_slot, x_perm, kept [E], dropped [E]), with room None
    (no limit) or the [E] per-expert room; experts(x_perm, offsets) -> y;
    combine(y, row_of_slot, w) -> out.  Returns out and the batch's
    statistics: counts, kept, dropped ([E] each) and the balance statistic.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    n = x.shape[0]
    idx, w, p = route(x)
    idx_np = np.asarray(idx.cpu() if hasattr(idx, "cpu") else idx, np.int64)
    counts = np.bincount(idx_np.reshape(-1), minlength=n_experts).astype(np.int64)
    # 2. the all-gather of every rank's counts and token count
    mine = torch.as_tensor(np.concatenate([counts, [n]]), dtype=torch.int64)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine, group=group)
    table = torch.stack(gathered).numpy()
    counts_all, n_global = table[:, :n_experts], int(table[:, n_experts].sum())
    cap = global_capacity(capacity_factor, n_global, n_experts)
    room = shard_room(counts_all, rank, cap)
    offsets, row_of_slot, x_perm, kept, dropped = dispatch(idx, x, room)
    y = experts(x_perm, offsets)
    out = combine(y, row_of_slot, w)
    # 5. the batch's statistics: counts and probability sums, kept, dropped
    p_np = np.asarray(p.cpu() if hasattr(p, "cpu") else p, np.float64)
    sums = torch.as_tensor(np.concatenate([counts, np.asarray(kept, np.int64),
                                           np.asarray(dropped, np.int64)]),
                           dtype=torch.int64)
    psum = torch.as_tensor(p_np.sum(axis=0), dtype=torch.float64)
    dist.all_reduce(sums, group=group)
    dist.all_reduce(psum, group=group)
    s = sums.numpy()
    e = n_experts
    stats = {"counts": s[:e], "kept": s[e:2 * e], "dropped": s[2 * e:],
             "balance": balance_statistic(s[:e], psum.numpy(), n_global, coef)}
    return out, stats
