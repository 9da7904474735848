"""Data parallelism with a capacity over the whole batch, with the library's
GPU stages.

"Expert Networks > Code Implementation" (In[10]) sets the capacity over the
batch, int(cf * (N // E)), and drops assignments in token order.  Two ranks
(processes, one CUDA context each) share the one device and hold
contiguous shards of unequal size.  Each rank routes its shard on the GPU
(moe_router_topk); routing_dispatch_expert_05_b300/dp.py all-gathers the
per-expert selection counts over gloo and gives each rank the room every
expert still has after the tokens before its shard; the rank then groups
with that per-expert room (moe_dispatch_permute_room), runs the grouped
FFN (moe_grouped_ffn) and combines (moe_combine).  A lock admits one rank's
GPU work at a time, so no kernel ever waits on another rank.

The kept/dropped sets must equal the whole batch's bit for bit, and the
outputs and balance statistic must match the oracle's layer on the whole
batch, fed the GPU's own logits (so near-ties cannot blur the drop sets).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu

WORLD = 2
SHARDS = (900, 1148)              # unequal shards of a 2048-token batch


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape():
    from routing_dispatch_expert_05_b300 import workloads as W
    # the capacity workload's layer (bf16 SiLU-MLP with biases, skewed
    # routing, cf 1.25) on 2048 tokens: capacity int(1.25 * 256) = 320
    return W.WORKLOADS["capacity_top2_bf16"].replace(name="dp_gpu", n_tokens=sum(SHARDS))


def _rank_main(rank, world, port, lock, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import dp
    from routing_dispatch_expert_05_b300 import moe as M
    from routing_dispatch_expert_05_b300 import workloads as W

    torch.cuda.set_device(0)
    shape = _shape()
    cuda = torch.device("cuda")
    with lock:
        t = M.upload(W.make_inputs(shape))
        torch.cuda.synchronize()
    d, E, k, F = shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    n = SHARDS[rank]
    s0 = sum(SHARDS[:rank])
    cfg = M.make_config(shape, n_tokens=n)
    # the grouping check of a shard's room-limited grouping: the shard's own
    # capacity is not the batch's, so it runs on a config without one
    cfg_check = M.make_config(shape.replace(capacity_factor=0.0), n_tokens=n)
    weights = M.make_weights(t)
    with lock:
        x = t["x"][s0:s0 + n].contiguous()
        ws = M.MoEWorkspace(cfg)
        torch.cuda.synchronize()
    keep = {}

    def route(xr):
        with lock:
            idx = torch.empty(n, k, dtype=torch.int32, device=cuda)
            w = torch.empty(n, k, dtype=torch.float32, device=cuda)
            lg = torch.empty(n, E, dtype=torch.float32, device=cuda)
            M.moe_router_topk(cfg, xr, weights, lg, idx, w, None, ws)
            torch.cuda.synchronize()
        keep["logits"] = lg.cpu().numpy()
        keep["idx"] = idx.cpu().numpy()
        keep["w"] = w.cpu().numpy()
        # the per-token probabilities of the statistic (the oracle's, on the
        # GPU's logits; test infrastructure)
        _, _, p = O.route(keep["logits"], shape.route, k)
        return idx, w, p

    def dispatch(idx, xr, room):
        assert room is not None
        with lock:
            rm = torch.as_tensor(np.asarray(room), dtype=torch.int32, device=cuda)
            offsets = torch.empty(E + 1, dtype=torch.int32, device=cuda)
            ros = torch.empty(n * k, dtype=torch.int32, device=cuda)
            tor = torch.empty(n * k, dtype=torch.int32, device=cuda)
            xp = torch.zeros(n * k, d, dtype=torch.bfloat16, device=cuda)
            kept = torch.empty(E, dtype=torch.int32, device=cuda)
            dropped = torch.empty(E, dtype=torch.int32, device=cuda)
            M.moe_dispatch_permute_room(cfg, idx, xr, rm, offsets, ros, tor, xp,
                                        M.make_stats(kept=kept, dropped=dropped), ws)
            M.moe_check_grouping(cfg_check, idx, offsets, ros, tor, ws)
            torch.cuda.synchronize()
            assert M.moe_read_device_error(ws) == M.MOE_OK
        keep["room"] = np.asarray(room).tolist()
        keep["row_of_slot"] = ros.cpu().numpy()
        return offsets, ros, xp, kept.cpu().numpy(), dropped.cpu().numpy()

    def experts(xp, offsets):
        with lock:
            h = torch.zeros(n * k, F, dtype=torch.bfloat16, device=cuda)
            y = torch.zeros(n * k, d, dtype=torch.float32, device=cuda)
            M.moe_grouped_ffn(cfg, xp, offsets, weights, h, y, ws)
            torch.cuda.synchronize()
        return y

    def combine(y, row_of_slot, w):
        with lock:
            o = torch.empty(n, d, dtype=torch.bfloat16, device=cuda)
            M.moe_combine(cfg, y, row_of_slot, w, None, o, ws)
            torch.cuda.synchronize()
            assert M.moe_read_device_error(ws) == M.MOE_OK
        return o

    got, stats = dp.dp_forward(x, route, dispatch, experts, combine, E,
                               shape.capacity_factor, shape.balance_coef)
    out[rank] = dict(out=got.float().cpu().numpy(), logits=keep["logits"], idx=keep["idx"],
                     w=keep["w"], row_of_slot=keep["row_of_slot"], room=keep["room"],
                     stats={key: np.asarray(v).tolist() if key != "balance" else float(v)
                            for key, v in stats.items()})
    dist.destroy_process_group()


def test_dp_capacity_over_the_batch_with_library_stages():
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import build as B
    from routing_dispatch_expert_05_b300 import workloads as W
    from tests.parity_util import BALANCE_REL, assert_output_close

    B.build()
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        lock = ctx.Lock()
        procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, lock, out))
                 for r in range(WORLD)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = {r: dict(out[r]) for r in range(WORLD)}
    shape = _shape()
    inp = W.make_inputs(shape)
    E, k = shape.n_experts, shape.top_k
    lg = np.concatenate([res[r]["logits"] for r in range(WORLD)])
    idx = np.concatenate([res[r]["idx"] for r in range(WORLD)])
    w = np.concatenate([res[r]["w"] for r in range(WORLD)]).astype(np.float64)
    # the whole batch's selection on the same logits is the ranks' selection
    i_o, w_o, p_o = O.route(lg, shape.route, k)
    assert np.array_equal(idx, i_o)
    # the whole batch's grouping: capacity over the batch, token order
    disp = O.dispatch(idx, E, float(np.float32(shape.capacity_factor)))
    assert disp["capacity"] == 320 and disp["dropped"].sum() > 0   # the cap does bind
    st = res[0]["stats"]
    assert st == res[1]["stats"]                          # every rank has the batch's
    for name in ("counts", "kept", "dropped"):
        assert np.array_equal(np.asarray(st[name]), disp[name]), name
    kept_mask = np.concatenate([res[r]["row_of_slot"] for r in range(WORLD)]) >= 0
    assert np.array_equal(kept_mask, disp["row_of_slot"] >= 0)
    assert res[1]["room"] != res[0]["room"]               # shard 1 had less room
    b_ref = O.balance_statistic(disp["counts"], p_o, shape.n_tokens, shape.balance_coef)
    assert abs(st["balance"] - b_ref) <= BALANCE_REL * abs(b_ref)
    # outputs: the oracle's experts on the whole batch's grouping, the GPU's weights
    x_perm = O.permute_rows(inp.values["x"], disp["token_of_row"])
    _, y = O.grouped_ffn(x_perm, disp["offsets"], inp.values, shape.expert, shape.dtype)
    exact = O.combine(y, disp["row_of_slot"], w)
    got = np.concatenate([res[r]["out"] for r in range(WORLD)])
    assert_output_close(got, exact, shape.dtype, "dp with batch capacity")
