"""Expert parallelism on CPU ranks (gloo): the exchange plan and the layer
forward with the experts sharded over 2 and 4 ranks.

Each rank routes and groups its own shard of the tokens, sends the rows to
the ranks holding their experts, runs only its own experts and gets the
outputs back (routing_dispatch_expert_05_b300/ep.py).  The per-rank stages here are the oracle's
(the exchange is what is under test); every token's output must equal the
single-process layer's.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from routing_dispatch_expert_05_b300 import ep  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_send_counts_are_contiguous_expert_blocks():
    offsets = [0, 3, 3, 7, 12, 12, 20]             # 6 experts
    c = ep.send_counts(offsets, 3)
    assert c.tolist() == [[3, 0], [4, 5], [0, 8]]
    with pytest.raises(ValueError):
        ep.send_counts(offsets, 4)


def test_receive_plan_is_the_expert_major_block_permutation():
    # 2 sources x 3 local experts; arrival order is source-major
    rc = np.array([[2, 0, 1], [1, 3, 0]])
    p = ep.receive_plan(rc)
    # arrival: s0e0 = [0, 1], s0e2 = [2], s1e0 = [3], s1e1 = [4, 5, 6]
    assert p.to_expert_major.tolist() == [0, 1, 3, 4, 5, 6, 2]
    assert p.local_offsets.tolist() == [0, 3, 6, 7]
    assert sorted(p.to_expert_major.tolist()) == list(range(7))
    assert p.rows_from.tolist() == [3, 4]


def _shape():
    from routing_dispatch_expert_05_b300 import workloads as W
    return W.MoEShape(name="ep", n_tokens=96, d_model=16, n_experts=8, top_k=3, d_ff=12,
                      expert=W.EXPERT_SWIGLU, route=W.ROUTE_TOPK_SOFTMAX, dtype=W.DTYPE_F32,
                      router_bias="normal", seed=9)


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import workloads as W
    shape = _shape()
    v = W.make_inputs(shape).values
    n = shape.n_tokens // world
    xs = v["x"][rank * n:(rank + 1) * n]

    def route(x):
        logits = O.router_logits(x, v["w_router"], v.get("b_router"))
        idx, w, _ = O.route(logits, shape.route, shape.top_k)
        return idx, w

    def dispatch(idx, x):
        d = O.dispatch(idx, shape.n_experts)
        return d["offsets"], d["row_of_slot"], torch.from_numpy(
            O.permute_rows(np.asarray(x, np.float64), d["token_of_row"]))

    def local_experts(rows, local_offsets, first):
        per = len(local_offsets) - 1
        p = {k: v[k][first:first + per] for k in ("w1", "w3", "w2")}
        _, y = O.grouped_ffn(rows.numpy(), local_offsets, p, shape.expert, shape.dtype)
        return torch.from_numpy(y)

    def combine(y_perm, row_of_slot, w):
        return O.combine(y_perm.numpy(), row_of_slot, w)

    got = ep.ep_forward(xs, route, dispatch, local_experts, combine, shape.n_experts)
    out[rank] = np.asarray(got).tolist()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_ep_forward_equals_single_process_layer(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(180)
            assert p.exitcode == 0
        res = dict(out)
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import workloads as W
    shape = _shape()
    ref = O.forward(shape, W.make_inputs(shape).values)["out_exact"]
    got = np.concatenate([np.asarray(res[r]) for r in range(world)])
    assert got.shape == ref.shape
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_receive_plan_properties_over_random_counts():
    """For any counts: the plan is a permutation of the arrival rows that
    visits experts in order, sources in order inside an expert, and each
    source's rows in arrival order; the group offsets are the per-expert
    totals."""
    hypothesis = pytest.importorskip("hypothesis")
    st = hypothesis.strategies

    @hypothesis.settings(max_examples=200, deadline=None)
    @hypothesis.given(st.integers(1, 4).flatmap(
        lambda r: st.integers(1, 5).flatmap(
            lambda l: st.lists(st.lists(st.integers(0, 6), min_size=l, max_size=l),
                               min_size=r, max_size=r))))
    def check(rows):
        rc = np.array(rows, np.int64)
        p = ep.receive_plan(rc)
        total = int(rc.sum())
        assert sorted(p.to_expert_major.tolist()) == list(range(total))
        assert p.local_offsets.tolist() == [0] + np.cumsum(rc.sum(axis=0)).tolist()
        assert p.rows_from.tolist() == rc.sum(axis=1).tolist()
        # label every arrival row with (expert, source, index within the block)
        labels = []
        for s in range(rc.shape[0]):
            for e in range(rc.shape[1]):
                labels += [(e, s, i) for i in range(rc[s, e])]
        ordered = [labels[a] for a in p.to_expert_major.tolist()]
        assert ordered == sorted(labels)

    check()


def test_send_counts_cover_the_grouped_buffer():
    rng = np.random.default_rng(12)
    for world in (1, 2, 4, 8):
        per_expert = rng.integers(0, 9, 16)
        offsets = np.concatenate([[0], np.cumsum(per_expert)])
        c = ep.send_counts(offsets, world)
        assert c.shape == (world, 16 // world)
        assert c.sum() == offsets[-1]
        # rank r's block is one contiguous slice of the grouped buffer
        starts = offsets[::16 // world][:world]
        assert (starts + c.sum(axis=1)).tolist() == offsets[16 // world::16 // world].tolist()
    assert list(ep.experts_of_rank(16, 4, 2)) == [8, 9, 10, 11]
