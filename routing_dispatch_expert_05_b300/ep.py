"""Expert parallelism: the exchange plan and the layer forward across ranks.

Expert parallelism ("DeepSeek 5.7: MoE from scratch", s.5: production
layers exchange tokens across expert-parallel devices; "Tutorial -- MoE SER
Expert Routing", configuration notes and next steps: experts sharded over
GPUs, an all-to-all dispatch) partitions the E routed experts contiguously
over R ranks: rank r holds
experts [r * E/R, (r+1) * E/R).  Every rank routes and groups its own tokens
exactly as the single-device layer does.  Because the grouped buffer is in
expert order and the experts are partitioned contiguously, the rows bound
for rank r are one contiguous block of it, so the send buffer of the first
exchange is the grouped buffer itself:

  1. dispatch locally (route, group by expert: offsets, row_of_slot, x_perm);
  2. exchange the per-(destination rank, expert) row counts (all-to-all);
  3. exchange the rows (all-to-all of x_perm blocks);
  4. the receiver holds, per source rank, rows grouped by its local experts;
     a block permutation brings them to expert-major order (expert, then
     source rank, then the source's order), the layout of one grouped
     problem over its local experts;
  5. run the local experts (grouped FFN), undo the block permutation;
  6. exchange the outputs back (the reverse all-to-all), which lands every
     output at its row of the sender's grouped buffer;
  7. combine locally with the sender's row_of_slot and weights.

The arithmetic per token is the single-device layer's, so the outputs are
identical for any R (the tests check that on CPU ranks).  Without a global
capacity the exchange carries everything; with one, the drop decision needs
the scan of counts over ranks before step 1's ranking and is not done here.

This module is the host side: the plan (pure index arithmetic) and the
orchestration over torch.distributed.  The per-rank stages are passed in as
callables -- on a GPU the library's own entry points (moe_router_topk,
moe_dispatch_permute, moe_grouped_ffn on the rank's slice of the expert
stacks, moe_combine) -- and the exchange is whatever backend the process
group has: NCCL between GPUs, or gloo through the host (whose all-to-all has
no 16-bit types, so bf16 rows travel as int32 pairs).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Sequence

import numpy as np


def experts_of_rank(n_experts: int, world_size: int, rank: int) -> range:
    """The contiguous block of experts rank `rank` holds."""
    if n_experts % world_size != 0:
        raise ValueError("expert parallelism needs E divisible by the number of ranks")
    per = n_experts // world_size
    return range(rank * per, (rank + 1) * per)


def send_counts(offsets: Sequence[int], world_size: int) -> np.ndarray:
    """Rows of the expert-sorted buffer bound for each rank: counts[r, e'] for
    r's local experts e' (shape [R, E/R]), from the local offsets [E+1]."""
    offsets = np.asarray(offsets, np.int64)
    per_expert = np.diff(offsets)
    n_experts = per_expert.shape[0]
    if n_experts % world_size != 0:
        raise ValueError("expert parallelism needs E divisible by the number of ranks")
    return per_expert.reshape(world_size, n_experts // world_size)


@dataclass
class ReceivePlan:
    """What a rank receives in the row exchange, in arrival order (source rank
    major, then its local-expert order), and how to regroup it."""
    recv_counts: np.ndarray      # [R, E/R] rows from source s for local expert e'
    to_expert_major: np.ndarray  # arrival index of each expert-major row
    local_offsets: np.ndarray    # [E/R + 1] expert-major group offsets

    @property
    def rows_from(self) -> np.ndarray:
        return self.recv_counts.sum(axis=1)


def receive_plan(recv_counts: np.ndarray) -> ReceivePlan:
    """The block permutation from arrival order (source-major) to expert-major
    order (expert, then source rank, then the source's row order)."""
    recv_counts = np.asarray(recv_counts, np.int64)
    n_src, n_local = recv_counts.shape
    # start of block (s, e') in arrival order
    arrive = np.zeros((n_src, n_local), np.int64)
    flat = recv_counts.reshape(-1)
    arrive.reshape(-1)[1:] = np.cumsum(flat)[:-1]
    order: List[np.ndarray] = []
    for e in range(n_local):
        for s in range(n_src):
            order.append(arrive[s, e] + np.arange(recv_counts[s, e], dtype=np.int64))
    perm = np.concatenate(order) if order else np.zeros(0, np.int64)
    local_offsets = np.zeros(n_local + 1, np.int64)
    local_offsets[1:] = np.cumsum(recv_counts.sum(axis=0))
    return ReceivePlan(recv_counts=recv_counts, to_expert_major=perm, local_offsets=local_offsets)


def ep_forward(x, route: Callable, dispatch: Callable, local_experts: Callable,
               combine: Callable, n_experts: int, group=None):
    """The layer forward for this rank's tokens x with the experts sharded.

    route(x) -> (idx, w); dispatch(idx, x) -> (offsets [E+1], row_of_slot,
    x_perm); local_experts(rows, local_offsets, first_expert) -> outputs of
    the local experts on expert-major rows; combine(y_perm, row_of_slot, w)
    -> out.  Rows and outputs are torch tensors on the process group's
    device (CPU for gloo, CUDA for NCCL).
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    idx, w = route(x)
    offsets, row_of_slot, x_perm = dispatch(idx, x)
    off_np = np.asarray(offsets.cpu() if hasattr(offsets, "cpu") else offsets, np.int64)
    sc = send_counts(off_np, world)                              # [R, E/R]
    send_c = torch.as_tensor(sc.reshape(-1), dtype=torch.int64)
    recv_c = torch.empty_like(send_c)
    dist.all_to_all_single(recv_c, send_c, group=group)          # counts per (src, e')
    plan = receive_plan(recv_c.reshape(world, -1).numpy())
    send_rows = sc.sum(axis=1).tolist()
    recv_rows = plan.rows_from.tolist()
    m_local = int(off_np[-1])
    d = x_perm.shape[1]
    rows_in = x_perm.new_empty((sum(recv_rows), d))
    dist.all_to_all_single(rows_in, x_perm[:m_local].contiguous(), recv_rows, send_rows,
                           group=group)
    perm = torch.as_tensor(plan.to_expert_major, dtype=torch.int64, device=rows_in.device)
    first = experts_of_rank(n_experts, world, rank).start
    y_sorted = local_experts(rows_in.index_select(0, perm), plan.local_offsets, first)
    y_arrival = torch.empty_like(y_sorted)
    y_arrival.index_copy_(0, perm, y_sorted)
    y_perm = y_sorted.new_empty((x_perm.shape[0], y_sorted.shape[1]))
    dist.all_to_all_single(y_perm[:m_local], y_arrival.contiguous(), send_rows, recv_rows,
                           group=group)
    return combine(y_perm, row_of_slot, w)
