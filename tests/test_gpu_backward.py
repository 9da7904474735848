"""GPU parity of the backward pass (moe_backward) against the backward
oracle.

The oracle differentiates in float64 without storage roundings; the GPU
path keeps its intermediates (g, u, h, dy, dh, [dg|du], dx_perm) in bf16
with fp32 accumulation.  A gradient passes
through about five such roundings, each within 2^-9 relative, so each
tensor is compared as ||gpu - oracle|| / ||oracle|| <= BWD_NORM (2e-2, a
few times the compounded rounding) and max |gpu - oracle| <= BWD_MAX *
max |oracle| (2e-2: no element far off; the products of Gaussian factors
these gradients are made of are heavy-tailed, so the bound scales with the
largest element, not the RMS).  The
routing the gradients are taken at is the GPU's own (read back with
moe_router_topk, the same kernels the backward recomputes it with), given
to the oracle, so a near-tie in the router cannot pick different experts on
the two sides.
"""
import numpy as np
import pytest
import torch

from oracle import moe_backward as OB
from oracle import moe_oracle as O
from routing_dispatch_expert_05_b300 import build as B
from routing_dispatch_expert_05_b300 import moe as M
from routing_dispatch_expert_05_b300 import workloads as W
from tests.parity_util import to_np

pytestmark = pytest.mark.gpu

BWD_NORM = 2e-2
BWD_MAX = 2e-2


def assert_grad_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), what
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / max(nrm, 1e-30)
    assert rel <= BWD_NORM, f"{what}: relative norm error {rel:.3e}"
    big = float(np.abs(ref).max())
    err = float(np.abs(got - ref).max())
    assert err <= BWD_MAX * big, f"{what}: max error {err:.3e} > {BWD_MAX} * {big:.3e}"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.load_library()
    torch.cuda.init()


def _shape(route, N=256, E=16, k=4, d=256, F=128, cf=0.0, router_bias="normal", seed=21,
           expert=W.EXPERT_SWIGLU, has_bias=False, n_shared=0, d_ff_shared=0):
    return W.MoEShape(name="bwd", n_tokens=N, d_model=d, n_experts=E, top_k=k, d_ff=F,
                      expert=expert, route=route, dtype=W.DTYPE_BF16, has_bias=has_bias,
                      router_bias=router_bias, sel_bias_range=0.1, capacity_factor=cf,
                      n_shared=n_shared, d_ff_shared=d_ff_shared, balance_coef=0.01, seed=seed)


def _grad_buffers(shape, inp):
    """NaN-filled fp32 gradient outputs for every parameter the layer has."""
    N, d, E, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.d_ff
    z = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")
    g = dict(dx=z(N, d), d_w_router=z(E, d), d_w1=z(E, F, d), d_w2=z(E, d, F))
    if shape.expert == W.EXPERT_SWIGLU:
        g["d_w3"] = z(E, F, d)
    if shape.has_bias:
        g["d_b1"] = z(E, F)
        g["d_b2"] = z(E, d)
    if shape.n_shared > 0:
        S, Fs = shape.n_shared, shape.d_ff_shared
        g.update(d_ws1=z(S, Fs, d), d_ws3=z(S, Fs, d), d_ws2=z(S, d, Fs))
    if "b_router" in inp.values:
        g["d_b_router"] = z(E)
    return g


GRAD_NAMES = ("dx", "d_w_router", "d_b_router", "d_w1", "d_w3", "d_w2", "d_b1", "d_b2",
              "d_ws1", "d_ws3", "d_ws2")


def _run(shape, d_balance, dout_seed=3):
    inp = W.make_inputs(shape)
    t = M.upload(inp)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    N, d, E, k, F = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k, shape.d_ff
    dout = np.random.default_rng(dout_seed).standard_normal((N, d)).astype(np.float32)
    dout = W.bits_to_f32(W.bf16_bits(dout))              # exactly representable in bf16
    dout_t = torch.from_numpy(dout).to(torch.bfloat16).cuda()
    g = _grad_buffers(shape, inp)
    grads = M.make_grads(**g)
    ws = M.MoEWorkspace(cfg, backward=True)
    M.moe_backward(cfg, t["x"], weights, dout_t, d_balance, grads, ws)
    # the routing the GPU recomputes, read back through the router entry point
    fws = M.MoEWorkspace(cfg)
    idx = torch.empty(N, k, dtype=torch.int32, device="cuda")
    w = torch.empty(N, k, dtype=torch.float32, device="cuda")
    M.moe_router_topk(cfg, t["x"], weights, None, idx, w, None, fws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == M.MOE_OK
    idx_np = to_np(idx).astype(np.int64)
    disp = O.dispatch(idx_np, E, shape.capacity_factor)
    kept = (disp["row_of_slot"] >= 0).reshape(idx_np.shape)
    ref = OB.layer_backward(shape, inp.values, dout, d_balance,
                            route_fixed=(idx_np, kept, disp["counts"]))
    return g, ref, ws, (cfg, t, weights, dout_t, grads)


CASES = [(W.ROUTE_SOFTMAX_TOPK, {}), (W.ROUTE_TOPK_SOFTMAX, dict(E=64, k=6)),
         (W.ROUTE_SIGMOID_BIAS, dict(E=32, k=3, router_bias="none")),
         (W.ROUTE_SOFTMAX_TOPK, dict(E=8, k=2, cf=1.0, N=320)),
         # enough rows per expert for the CTA-pair GEMMs
         (W.ROUTE_TOPK_SOFTMAX, dict(N=2048)),
         # SiLU-MLP experts with biases ("Expert Networks", In[7]), with a
         # capacity that drops; and without biases
         (W.ROUTE_SOFTMAX_TOPK, dict(E=8, k=2, N=320, cf=1.25, expert=W.EXPERT_SILU_MLP,
                                     has_bias=True)),
         (W.ROUTE_TOPK_SOFTMAX, dict(E=16, k=4, expert=W.EXPERT_SILU_MLP)),
         # shared SwiGLU experts beside sigmoid routing ("DeepSeek 5.7", s.4),
         # one and two of them, CTA pairs for the latter
         (W.ROUTE_SIGMOID_BIAS, dict(E=16, k=4, router_bias="none", n_shared=1,
                                     d_ff_shared=128)),
         (W.ROUTE_SIGMOID_BIAS, dict(E=32, k=6, N=1024, router_bias="none", n_shared=2,
                                     d_ff_shared=64)),
         # widths over several 256-wide weight-gradient tiles with ragged
         # edges (d = 384, F = 320: the dW1 / dW3 split inside a tile)
         (W.ROUTE_SOFTMAX_TOPK, dict(N=1024, E=8, k=2, d=384, F=320)),
         (W.ROUTE_SIGMOID_BIAS, dict(N=512, E=8, k=2, d=320, F=192, router_bias="none",
                                     n_shared=1, d_ff_shared=320))]


@pytest.mark.parametrize("d_balance", [0.0, 0.7])
@pytest.mark.parametrize("route,kw", CASES)
def test_backward_matches_oracle(route, kw, d_balance):
    shape = _shape(route, **kw)
    g, ref, _, _ = _run(shape, d_balance)
    for name in GRAD_NAMES:
        if name not in g:
            continue
        assert_grad_close(to_np(g[name]), ref[name], name)


@pytest.mark.parametrize("k", [2, 8])
def test_backward_worked_example(k):
    """"DeepSeek 5.7", Worked example: B = 2, T = 4, top-2 routing, one shared
    expert; router gradients exist, experts no token selected receive no
    gradient, and with top-k over every expert the layer is the dense
    all-expert sum.  At the nearest size the tensor-core backward tiles: d = 64
    (the page: 16), 8 routed experts (the page: 4), F = Fs = 64; SwiGLU
    experts, sigmoid routing with a selection bias.  k = 8 is the dense case
    (every expert selected)."""
    shape = _shape(W.ROUTE_SIGMOID_BIAS, N=8, E=8, k=k, d=64, F=64, router_bias="none",
                   n_shared=1, d_ff_shared=64, seed=5)
    g, ref, _, _ = _run(shape, 0.3)
    for name in GRAD_NAMES:
        if name in g:
            assert_grad_close(to_np(g[name]), ref[name], name)
    # router gradients exist
    assert float(g["d_w_router"].abs().max()) > 0
    # each token has exactly k routed assignments; experts no token chose
    # receive exact zeros
    inp = W.make_inputs(shape)
    idx, _, _ = OB.fixed_route(shape, inp.values)
    assert idx.shape == (8, k) and all(len(set(r)) == k for r in idx.tolist())
    unused = sorted(set(range(8)) - set(idx.reshape(-1).tolist()))
    if k == 2:
        assert unused, "8 tokens x 2 slots left every expert chosen"
    for e in unused:
        for name in ("d_w1", "d_w3", "d_w2"):
            assert torch.count_nonzero(g[name][e]) == 0, (name, e)


def test_backward_unused_expert_gets_zero():
    shape = _shape(W.ROUTE_SOFTMAX_TOPK, N=128, E=16, k=2)
    inp = W.make_inputs(shape)
    assert "b_router" in inp.values
    inp.values["b_router"][5] = -60.0                     # nobody selects expert 5
    inp.bits["b_router"] = W.bf16_bits(inp.values["b_router"])
    t = M.upload(inp)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    N, d = shape.n_tokens, shape.d_model
    dout = torch.randn(N, d, device="cuda").to(torch.bfloat16)
    g = _grad_buffers(shape, inp)
    ws = M.MoEWorkspace(cfg, backward=True)
    M.moe_backward(cfg, t["x"], weights, dout, 0.0, M.make_grads(**g), ws)
    torch.cuda.synchronize()
    for name in ("d_w1", "d_w3", "d_w2"):
        assert torch.count_nonzero(g[name][5]) == 0, name
        assert torch.isfinite(g[name]).all(), name


def test_backward_is_deterministic():
    shape = _shape(W.ROUTE_TOPK_SOFTMAX, E=64, k=6)
    g, _, ws, (cfg, t, weights, dout_t, grads) = _run(shape, 0.5)
    first = {k_: v.clone() for k_, v in g.items()}
    M.moe_backward(cfg, t["x"], weights, dout_t, 0.5, grads, ws)
    torch.cuda.synchronize()
    for name, v in g.items():
        assert torch.equal(v, first[name]), name


@pytest.mark.parametrize("name", ["qwen3_moe", "deepseek_v3_block"])
def test_backward_full_size_sampled(name):
    """A full-size layer -- Qwen3-style (16384 tokens, 128 experts, top-8,
    the skewed grouping of the workload: 2 to ~16,000 rows per expert) or
    DeepSeek-style (8192 tokens, 64 experts, top-6, sigmoid routing with a
    selection bias, two shared experts) -- the backward as the bench times
    it, checked on samples the oracle computes exactly from the GPU's own
    routing:
    - dx of 16 tokens: with d_balance = 0 a token's input gradient depends on
      that token alone, so the oracle runs on those tokens;
    - the weight gradients of two experts (the smallest of at least 20
      rows, and one of a few hundred): an expert's gradient sums over the
      assignments routed to it, so the oracle runs on exactly the tokens
      that chose it, with every other assignment of theirs marked as not
      kept (their routing weights still normalise over all of a token's
      selected logits)."""
    shape = W.WORKLOADS[name]
    assert shape.expert == W.EXPERT_SWIGLU and not shape.has_bias
    inp = W.make_inputs(shape)
    t = M.upload(inp)
    cfg = M.make_config(shape)
    weights = M.make_weights(t)
    N, d, E, k = shape.n_tokens, shape.d_model, shape.n_experts, shape.top_k
    dout = np.random.default_rng(11).standard_normal((N, d)).astype(np.float32)
    dout = W.bits_to_f32(W.bf16_bits(dout))
    dout_t = torch.from_numpy(dout).to(torch.bfloat16).cuda()
    g = _grad_buffers(shape, inp)
    ws = M.MoEWorkspace(cfg, backward=True)
    M.moe_backward(cfg, t["x"], weights, dout_t, 0.0, M.make_grads(**g), ws)
    fws = M.MoEWorkspace(cfg)
    idx = torch.empty(N, k, dtype=torch.int32, device="cuda")
    w = torch.empty(N, k, dtype=torch.float32, device="cuda")
    M.moe_router_topk(cfg, t["x"], weights, None, idx, w, None, fws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(ws) == M.MOE_OK
    idx_np = to_np(idx).astype(np.int64)
    disp = O.dispatch(idx_np, E, shape.capacity_factor)
    kept = (disp["row_of_slot"] >= 0).reshape(idx_np.shape)
    counts = disp["counts"]

    def oracle_on(tokens, kept_sub):
        vals = dict(inp.values)
        vals["x"] = inp.values["x"][tokens]
        sub = shape.replace(n_tokens=len(tokens))
        return OB.layer_backward(sub, vals, dout[tokens], 0.0,
                                 route_fixed=(idx_np[tokens], kept_sub, counts))

    toks = np.sort(np.random.default_rng(5).choice(N, 16, replace=False))
    ref = oracle_on(toks, kept[toks])
    assert_grad_close(to_np(g["dx"])[toks], ref["dx"], "dx (16 sampled tokens)")
    del ref

    rows = counts.astype(np.int64)
    # the smallest expert of at least 20 rows, and one of a few hundred
    cand = np.nonzero(rows >= 20)[0]
    small = int(cand[np.argmin(rows[cand])])
    medium = int(np.nonzero((rows >= 200) & (rows <= 600))[0][0])
    for e in (small, medium):
        tok_e = np.nonzero((idx_np == e).any(axis=1))[0]
        kept_e = kept[tok_e] & (idx_np[tok_e] == e)
        ref = oracle_on(tok_e, kept_e)
        for name in ("d_w1", "d_w3", "d_w2"):
            assert_grad_close(to_np(g[name][e]), ref[name][e], f"{name}[{e}] ({rows[e]} rows)")
        del ref
