"""Data parallelism with a capacity over the whole batch, on CPU ranks (gloo).

The token shards of the batch go to 2, 3 (shards of unequal size) and 4 ranks.  Each rank routes its own
tokens, the all-gathered per-expert counts give it the room each expert
still has after the tokens before its shard
(routing_dispatch_expert_05_b300/dp.py), and it groups, runs the experts and
combines its own shard.  The per-rank stages are the oracle's; the exchange
is what is under test.  Every token's output, the kept and dropped counts
and the balance statistic must equal those of the layer run on the whole
batch at once.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from routing_dispatch_expert_05_b300 import dp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape(n_tokens=256, cf=1.25):
    from routing_dispatch_expert_05_b300 import workloads as W
    # the capacity workload's layer (SiLU-MLP with biases, skewed routing,
    # cf 1.25), smaller: capacity int(1.25 * (256 // 8)) = 40 per expert
    return W.WORKLOADS["capacity_top2_fp32"].replace(name="dp", n_tokens=n_tokens, d_model=32,
                                                     d_ff=48, capacity_factor=cf)


def test_shard_room_is_what_the_batch_rule_leaves():
    counts_all = np.array([[5, 0, 9], [3, 4, 1], [7, 7, 7]])
    assert dp.prior_counts(counts_all, 0).tolist() == [0, 0, 0]
    assert dp.prior_counts(counts_all, 2).tolist() == [8, 4, 10]
    assert dp.shard_room(counts_all, 0, 6).tolist() == [6, 6, 6]
    assert dp.shard_room(counts_all, 1, 6).tolist() == [1, 6, 0]
    assert dp.shard_room(counts_all, 2, 6).tolist() == [0, 2, 0]
    assert dp.shard_room(counts_all, 2, None) is None
    assert dp.global_capacity(1.25, 256, 8) == 40
    assert dp.global_capacity(1.25, 11, 4) == 2          # int(1.25 * 2)
    assert dp.global_capacity(0.0, 256, 8) is None


def test_shard_rooms_reproduce_the_batch_drop_set():
    """Without processes: per-shard grouping with the shard rooms keeps
    exactly the assignments the batch-wide token-order rule keeps."""
    from oracle import moe_oracle as O
    rng = np.random.default_rng(8)
    E, k = 6, 2
    for world in (2, 3, 4):
        for cf in (0.5, 1.0, 1.5):
            n = 30
            idx = np.stack([rng.choice(E, k, replace=False, p=[.4, .2, .15, .1, .1, .05])
                            for _ in range(n * world)])
            whole = O.dispatch(idx, E, cf)
            cap = dp.global_capacity(cf, n * world, E)
            shards = idx.reshape(world, n, k)
            counts_all = np.stack([np.bincount(s.reshape(-1), minlength=E) for s in shards])
            kept_mask = []
            for r in range(world):
                d = O.dispatch(shards[r], E, expert_capacity=dp.shard_room(counts_all, r, cap))
                kept_mask.append(d["row_of_slot"] >= 0)
            assert np.array_equal(np.concatenate(kept_mask), whole["row_of_slot"] >= 0)


def _shard(n_tokens, world, rank):
    """Contiguous shards; with 3 ranks they differ in size (85, 85, 86)."""
    bounds = [n_tokens * r // world for r in range(world + 1)]
    return bounds[rank], bounds[rank + 1]


def _rank_main(rank, world, port, cf, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import workloads as W
    shape = _shape(cf=cf)
    v = W.make_inputs(shape).values
    lo, hi = _shard(shape.n_tokens, world, rank)
    xs = v["x"][lo:hi]

    def route(x):
        logits = O.router_logits(x, v["w_router"], v.get("b_router"))
        return O.route(logits, shape.route, shape.top_k)

    def dispatch(idx, x, room):
        d = O.dispatch(idx, shape.n_experts, expert_capacity=room) if room is not None \
            else O.dispatch(idx, shape.n_experts)
        x_perm = O.permute_rows(np.asarray(x, np.float64), d["token_of_row"])
        return d["offsets"], d["row_of_slot"], x_perm, d["kept"], d["dropped"]

    def experts(x_perm, offsets):
        return O.grouped_ffn(x_perm, offsets, v, shape.expert, shape.dtype)[1]

    def combine(y, row_of_slot, w):
        return O.combine(y, row_of_slot, w)

    got, stats = dp.dp_forward(xs, route, dispatch, experts, combine, shape.n_experts,
                               shape.capacity_factor, shape.balance_coef)
    out[rank] = (np.asarray(got).tolist(), {k: (np.asarray(s).tolist()
                                                 if k != "balance" else s)
                                            for k, s in stats.items()})
    dist.destroy_process_group()


@pytest.mark.parametrize("world,cf", [(2, 1.25), (3, 1.25), (4, 1.25), (2, 0.0)])
def test_dp_forward_with_batch_capacity_equals_the_whole_batch(world, cf):
    """cf 0: no capacity, the ranks are plain replicas and nothing drops."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, cf, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import workloads as W
    shape = _shape(cf=cf)
    ref = O.forward(shape, W.make_inputs(shape).values)
    assert (ref["dropped"].sum() > 0) == (cf > 0)         # the capacity binds
    got = np.concatenate([np.asarray(res[r][0]) for r in range(world)])
    assert np.allclose(got, ref["out_exact"], rtol=1e-12, atol=1e-12)
    for r in range(world):
        stats = res[r][1]
        assert stats["counts"] == ref["counts"].tolist()
        assert stats["kept"] == ref["kept"].tolist()
        assert stats["dropped"] == ref["dropped"].tolist()
        assert stats["balance"] == pytest.approx(ref["balance"], rel=1e-12)
    # each shard on its own capacity int(cf * (n // E)) would keep another set
    # of assignments (the exchange is needed)
    if cf > 0:
        local = [O.dispatch(ref["idx"][slice(*_shard(shape.n_tokens, world, r))],
                            shape.n_experts, shape.capacity_factor)["row_of_slot"] >= 0
                 for r in range(world)]
        assert not np.array_equal(np.concatenate(local), ref["row_of_slot"] >= 0)
