"""Expert parallelism with the library's own stages on the GPU.

Two ranks (processes, one CUDA context each) share the one device; each
holds half of the experts.  Every GPU step is the library's: the router and
selection (moe_router_topk), the grouping (moe_dispatch_permute), the
grouped SwiGLU FFN of the rank's own experts (moe_grouped_ffn on the
received, expert-major rows with weight pointers into its slice of the
stacks) and the weighted combine (moe_combine).  The exchange plan and the
all-to-alls are routing_dispatch_expert_05_b300/ep.py over gloo, so the
exchange runs on the host: no rank's kernel ever waits on another rank.  A
lock shared by the ranks admits one rank's GPU work at a time (each stage
ends with a synchronize before the lock is released), so the two contexts
never execute at once.  Each rank's output must match the oracle's layer on
its tokens.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape():
    from routing_dispatch_expert_05_b300 import workloads as W
    return W.MoEShape(name="ep_gpu", n_tokens=1024, d_model=256, n_experts=16, top_k=4,
                      d_ff=192, expert=W.EXPERT_SWIGLU, route=W.ROUTE_TOPK_SOFTMAX,
                      dtype=W.DTYPE_BF16, router_bias="none", seed=31)


def _rank_main(rank, world, port, lock, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from routing_dispatch_expert_05_b300 import ep
    from routing_dispatch_expert_05_b300 import moe as M
    from routing_dispatch_expert_05_b300 import workloads as W

    torch.cuda.set_device(0)
    shape = _shape()
    with lock:
        t = M.upload(W.make_inputs(shape))
        torch.cuda.synchronize()
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    n = N // world
    cuda = torch.device("cuda")
    cfg = M.make_config(shape, n_tokens=n)
    weights = M.make_weights(t)
    with lock:
        x = t["x"][rank * n:(rank + 1) * n].contiguous()
        ws = M.MoEWorkspace(cfg)
        torch.cuda.synchronize()

    def route(xr):
        with lock:
            idx = torch.empty(n, k, dtype=torch.int32, device=cuda)
            w = torch.empty(n, k, dtype=torch.float32, device=cuda)
            M.moe_router_topk(cfg, xr, weights, None, idx, w, None, ws)
            torch.cuda.synchronize()
        return idx, w

    def dispatch(idx, xr):
        with lock:
            offsets = torch.empty(E + 1, dtype=torch.int32, device=cuda)
            ros = torch.empty(n * k, dtype=torch.int32, device=cuda)
            tor = torch.empty(n * k, dtype=torch.int32, device=cuda)
            xp = torch.zeros(n * k, d, dtype=torch.bfloat16, device=cuda)
            M.moe_dispatch_permute(cfg, idx, xr, offsets, ros, tor, xp, None, ws)
            torch.cuda.synchronize()
        # rows travel through the host as their bit patterns, two bf16 per
        # int32 (gloo's all-to-all has no 16-bit types)
        return offsets.cpu(), ros, xp.cpu().view(torch.int32)

    def local_experts(rows, local_offsets, first):
        per = len(local_offsets) - 1
        m = rows.shape[0]
        # buffers sized for the most rows this rank can receive: every token
        # of every rank, k rows each
        lcfg = M.make_config(shape.replace(n_experts=per))
        lw = M.make_weights({name: t[name][first:first + per] for name in ("w1", "w3", "w2")})
        assert 0 <= m <= N * k and int(local_offsets[-1]) == m
        with lock:
            lws = M.MoEWorkspace(lcfg)
            xr = torch.zeros(N * k, d, dtype=torch.bfloat16, device=cuda)
            xr[:m] = rows.to(cuda).view(torch.bfloat16)      # [m, d / 2] int32 -> [m, d]
            offs = torch.as_tensor(np.asarray(local_offsets), dtype=torch.int32, device=cuda)
            h = torch.zeros(N * k, F, dtype=torch.bfloat16, device=cuda)
            y = torch.zeros(N * k, d, dtype=torch.float32, device=cuda)
            M.moe_grouped_ffn(lcfg, xr, offs, lw, h, y, lws)
            torch.cuda.synchronize()
            assert M.moe_read_device_error(lws) == M.MOE_OK
            return y[:m].cpu()

    def combine(y_perm, row_of_slot, w):
        with lock:
            o = torch.empty(n, d, dtype=torch.bfloat16, device=cuda)
            M.moe_combine(cfg, y_perm.to(cuda), row_of_slot, w, None, o, ws)
            torch.cuda.synchronize()
        return o

    got = ep.ep_forward(x, route, dispatch, local_experts, combine, E)
    with lock:
        assert M.moe_read_device_error(ws) == M.MOE_OK
        out[rank] = got.float().cpu().numpy().tolist()
    dist.destroy_process_group()


def test_ep_forward_with_library_stages_matches_oracle():
    from oracle import moe_oracle as O
    from routing_dispatch_expert_05_b300 import build as B
    from routing_dispatch_expert_05_b300 import workloads as W
    from tests.parity_util import assert_output_close, set_ambiguous_tokens

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
        res = dict(out)
    shape = _shape()
    inp = W.make_inputs(shape)
    got = np.concatenate([np.asarray(res[r]) for r in range(WORLD)])
    ref = O.forward(shape, inp.values)
    keys = O.selection_keys(ref["logits"], shape.route)
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, 4e-4)
    assert amb.mean() < 0.05
    assert_output_close(got[~amb], ref["out_exact"][~amb], shape.dtype, "ep")
