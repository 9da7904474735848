"""The allocation-free grouping entry point against the workspace one.

moe_dispatch_permute_noalloc serves callers that cannot give the library any
device memory of its own -- a serving engine that has already claimed the
GPU's memory for its pool, or a hot loop that must not call cudaMalloc
because it can stall the device.  It keeps the per-chunk histogram in a
fixed array inside the library, so it must produce exactly what
moe_dispatch_permute produces with a workspace: same offsets, rows, tokens,
copied rows and counts, bit for bit, call after call (the shared array keeps
the previous call's contents).

This file is collected last on purpose and builds its own library handle, so
it runs the same alone in a fresh process or after every other test.
"""
import ctypes

import pytest
import torch

from routing_dispatch_expert_05_b300 import build as B
from routing_dispatch_expert_05_b300 import moe as M
from routing_dispatch_expert_05_b300 import workloads as W

pytestmark = pytest.mark.gpu


def _shape(n_tokens, n_experts, top_k, cf, dtype):
    return W.MoEShape(name="noalloc", n_tokens=n_tokens, d_model=256, n_experts=n_experts,
                      top_k=top_k, d_ff=64, expert=W.EXPERT_SWIGLU,
                      route=W.ROUTE_SOFTMAX_TOPK, dtype=dtype, capacity_factor=cf)


def _run(fn_ws, shape, idx, x):
    """Outputs of one grouping call (fn_ws True: with a workspace)."""
    cfg = M.make_config(shape)
    N, E, k, d = shape.n_tokens, shape.n_experts, shape.top_k, shape.d_model
    o = dict(offsets=torch.full((E + 1,), -5, dtype=torch.int32, device="cuda"),
             ros=torch.full((N * k,), -5, dtype=torch.int32, device="cuda"),
             tor=torch.full((N * k,), -5, dtype=torch.int32, device="cuda"),
             xp=torch.zeros(N * k, d, dtype=x.dtype, device="cuda"),
             counts=torch.full((E,), -5, dtype=torch.int32, device="cuda"),
             kept=torch.full((E,), -5, dtype=torch.int32, device="cuda"),
             dropped=torch.full((E,), -5, dtype=torch.int32, device="cuda"))
    stats = M.make_stats(counts=o["counts"], kept=o["kept"], dropped=o["dropped"])
    if fn_ws:
        ws = M.MoEWorkspace(cfg, forward=False)
        M.moe_dispatch_permute(cfg, idx, x, o["offsets"], o["ros"], o["tor"], o["xp"],
                               stats, ws)
    else:
        M.moe_dispatch_permute_noalloc(cfg, idx, x, o["offsets"], o["ros"], o["tor"],
                                       o["xp"], stats)
    torch.cuda.synchronize()
    return o


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.load_library()


CASES = [  # (tokens, experts, k, capacity factor, dtype, Zipf skew)
    (4096, 8, 2, 1.25, W.DTYPE_BF16, 1.1),
    (5000, 128, 8, 0.0, W.DTYPE_BF16, 1.1),
    (777, 64, 6, 1.0, W.DTYPE_F32, 0.0),
]


def test_noalloc_dispatch_matches_workspace_dispatch_twice_in_a_row():
    for n, e, k, cf, dt, zipf in CASES:
        shape = _shape(n, e, k, cf, dt)
        x = torch.randn(n, shape.d_model, device="cuda").to(M.torch_dtype(dt))
        for call, seed in enumerate((11, 12)):     # two calls in a row, new inputs
            idx = torch.from_numpy(W.make_assignments(n, e, k, seed=seed + n,
                                                      zipf_s=zipf)).cuda()
            ref = _run(True, shape, idx, x)
            got = _run(False, shape, idx, x)
            m = int(ref["offsets"][-1])
            for key in ("offsets", "ros", "counts", "kept", "dropped"):
                assert torch.equal(got[key], ref[key]), (n, e, call, key)
            assert torch.equal(got["tor"][:m], ref["tor"][:m]), (n, e, call)
            assert torch.equal(got["xp"][:m], ref["xp"][:m]), (n, e, call)


def test_noalloc_dispatch_rejects_more_tokens_than_its_array_holds():
    lib = M.load_library()
    cfg = M.make_config(_shape(65537, 8, 2, 0.0, W.DTYPE_BF16))
    buf = torch.zeros(1024, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    st = lib.moe_dispatch_permute_noalloc(ctypes.byref(cfg), p, None, p, p, p, None,
                                          None, None)
    assert st == M.MOE_ERR_UNSUPPORTED
