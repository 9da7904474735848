"""Parity of every stage of the CUDA path with the CPU oracle, on identical
seeded inputs, through the C ABI.  Sizes span several tiles and end in a
ragged tail; edge cases cover empty experts, N < E, k = E, E = 1, N = 0 and
capacity drops."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_05_b300 import build as B
from routing_dispatch_expert_05_b300 import moe as M
from routing_dispatch_expert_05_b300 import workloads as W
from tests.parity_util import (BALANCE_REL, Device, ambiguous_tokens,
                               assert_close_rms, assert_output_close,
                               assert_within_ulp,
                               check_selection_valid, dev, inputs_for,
                               logit_margin, rel_tol, set_ambiguous_tokens,
                               to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.load_library()
    torch.cuda.init()


def _cfg(**kw):
    base = dict(name="t", n_tokens=100, d_model=64, n_experts=8, top_k=2, d_ff=64,
                expert=W.EXPERT_SWIGLU, route=W.ROUTE_SOFTMAX_TOPK,
                dtype=W.DTYPE_F32)
    base.update(kw)
    return W.MoEShape(**base)


# ------------------------------------------------ selection from logits
ROUTE_CASES = [(8, 2), (5, 3), (33, 4), (64, 6), (128, 8), (256, 8), (8, 8),
               (1, 1), (200, 1), (40, 40)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("E,k", ROUTE_CASES)
@pytest.mark.parametrize("kind", ["normal", "ties", "signed_zero"])
def test_route_logits_bit_exact(mode, E, k, kind):
    N = 1000
    seed = 1000 * mode + 10 * E + k
    logits = W.make_logits(N, E, seed=seed, kind=kind)
    bias = np.random.default_rng(seed).uniform(-0.1, 0.1, E).astype(np.float32) \
        if mode == 2 else None
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, route=mode)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    idx = torch.full((N, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((N, k), dtype=torch.float32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    bal = torch.zeros(1, dtype=torch.float32, device="cuda")
    M.moe_route_logits(cfg, dev(logits), dev(bias) if bias is not None else None,
                       idx, w, M.make_stats(counts=counts, balance=bal), ws)
    torch.cuda.synchronize()
    i_o, w_o, p_o = O.route(logits, mode, k, bias)
    assert np.array_equal(to_np(idx), i_o)
    assert np.allclose(to_np(w), w_o, rtol=2e-6, atol=2e-7)
    cnt_o = np.bincount(i_o.reshape(-1), minlength=E)
    assert np.array_equal(to_np(counts), cnt_o)
    b_o = O.balance_statistic(cnt_o, p_o, N, shape.balance_coef)
    assert abs(float(to_np(bal)[0]) - b_o) <= BALANCE_REL * abs(b_o)
    assert M.moe_read_device_error(ws) == M.MOE_OK


def test_route_logits_empty_and_tail():
    for N in (0, 1, 127, 129):
        shape = _cfg(n_tokens=N, n_experts=16, top_k=4)
        cfg = M.make_config(shape)
        ws = M.MoEWorkspace(cfg, forward=False)
        logits = W.make_logits(max(N, 1), 16, seed=N)[:N]
        idx = torch.full((max(N, 1), 4), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((max(N, 1), 4), dtype=torch.float32, device="cuda")
        counts = torch.full((16,), 5, dtype=torch.int32, device="cuda")
        bal = torch.full((1,), 5.0, device="cuda")
        lg = dev(logits) if N else torch.zeros(16, device="cuda")
        M.moe_route_logits(cfg, lg, None, idx, w, M.make_stats(counts=counts, balance=bal), ws)
        torch.cuda.synchronize()
        i_o, _, _ = O.route(logits, 0, 4) if N else (np.zeros((0, 4)), None, None)
        assert np.array_equal(to_np(idx)[:N], i_o)
        assert to_np(counts).sum() == 4 * N
        if N == 0:
            assert float(to_np(bal)[0]) == 0.0


# ------------------------------------------------------------- dispatch
DISPATCH_CASES = [
    # N, E, k, capacity_factor, zipf
    (1000, 8, 2, 1.25, 0.0),
    (1000, 8, 2, 0.0, 0.0),
    (777, 64, 6, 0.0, 1.1),
    (4096, 8, 2, 1.25, 1.5),
    (3, 8, 2, 1.25, 0.0),      # N < E: capacity 0, everything dropped
    (1, 1, 1, 0.0, 0.0),       # E = 1
    (300, 16, 16, 0.0, 0.0),   # k = E
    (513, 128, 8, 0.0, 1.1),   # many empty experts
    (2000, 256, 4, 2.0, 1.2),
    (600, 7, 3, 1.0, 0.8),
]


@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("N,E,k,cf,zipf", DISPATCH_CASES)
def test_dispatch_bit_exact(N, E, k, cf, zipf, dtype):
    d = 64
    idx = W.make_assignments(N, E, k, seed=N + E + k, zipf_s=zipf)
    x = np.random.default_rng(N).standard_normal((N, d)).astype(np.float32)
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d, capacity_factor=cf,
                 dtype=dtype)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    td = M.torch_dtype(dtype)
    xd = dev(x, dtype)
    offsets = torch.full((E + 1,), -5, dtype=torch.int32, device="cuda")
    ros = torch.full((N * k,), -5, dtype=torch.int32, device="cuda")
    tor = torch.full((N * k,), -5, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((N * k, d), dtype=td, device="cuda")
    st = {n: torch.full((E,), -5, dtype=torch.int32, device="cuda")
          for n in ("counts", "kept", "dropped")}
    M.moe_dispatch_permute(cfg, dev(idx), xd, offsets, ros, tor, x_perm,
                           M.make_stats(**st), ws)
    torch.cuda.synchronize()
    # the config stores capacity_factor as fp32; the oracle gets the same value
    res = O.dispatch(idx, E, float(np.float32(cf)))
    assert np.array_equal(to_np(offsets), res["offsets"])
    assert np.array_equal(to_np(ros), res["row_of_slot"])
    m = int(res["offsets"][-1])
    assert np.array_equal(to_np(tor)[:m], res["token_of_row"])
    for n in ("counts", "kept", "dropped"):
        assert np.array_equal(to_np(st[n]), res[n]), n
    got = x_perm[:m].view(torch.int16 if dtype == W.DTYPE_BF16 else torch.int32)
    ref = xd[torch.from_numpy(res["token_of_row"]).cuda()].view(got.dtype) if m else got
    assert torch.equal(got, ref)
    assert M.moe_read_device_error(ws) == M.MOE_OK


def test_dispatch_flags_bad_expert_index():
    N, E, k, d = 64, 8, 2, 32
    idx = W.make_assignments(N, E, k, seed=3)
    idx[5, 1] = 8       # out of range
    idx[9, 0] = -1      # out of range
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    x = torch.randn(N, d, device="cuda")
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.zeros(N * k, dtype=torch.int32, device="cuda")
    tor = torch.zeros(N * k, dtype=torch.int32, device="cuda")
    xp = torch.zeros(N * k, d, device="cuda")
    M.moe_dispatch_permute(cfg, dev(idx), x, offsets, ros, tor, xp, None, ws)
    assert M.moe_read_device_error(ws) == M.MOE_ERR_DEVICE_CHECK
    assert M.moe_read_device_error(ws) == M.MOE_OK      # read clears it
    r = to_np(ros)
    assert r[5 * k + 1] == -1 and r[9 * k + 0] == -1
    assert int(to_np(offsets)[-1]) == N * k - 2


# ---------------------------------------------------------- expert FFNs
FFN_CASES = [("toy_top2_fp32", 64), ("capacity_top2_fp32", 700),
             ("capacity_top2_bf16", 700), ("deepseek_v3_block", 300),
             ("qwen3_moe", 200),
             # enough rows per expert for CTA pairs, with short group tails
             # left to the single-CTA pass
             ("deepseek_v3_block", 1536)]


def _oracle_dispatch_inputs(shape, inp, zipf=1.1, seed=77):
    idx = W.make_assignments(shape.n_tokens, shape.n_experts, shape.top_k, seed=seed,
                             zipf_s=zipf)
    disp = O.dispatch(idx, shape.n_experts, float(np.float32(shape.capacity_factor)))
    x_perm = O.permute_rows(inp.values["x"], disp["token_of_row"])
    return idx, disp, x_perm


def _padded(a, rows):
    out = np.zeros((rows,) + a.shape[1:], a.dtype)
    out[:a.shape[0]] = a
    return out


@pytest.mark.parametrize("name,N", FFN_CASES)
def test_expert_up_down_parity(name, N):
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    _, disp, x_perm = _oracle_dispatch_inputs(shape, inp)
    h_o, y_o = O.grouped_ffn(x_perm, disp["offsets"], inp.values, shape.expert,
                             shape.dtype)
    rows = shape.n_tokens * shape.top_k
    m = int(disp["offsets"][-1])
    xp = dev(_padded(x_perm.astype(np.float32), rows), shape.dtype)
    off = dev(disp["offsets"].astype(np.int32))
    h = D.empty(rows, shape.d_ff)
    M.moe_expert_up(D.cfg, xp, off, D.weights, h, D.ws)
    # down on the oracle's h, so the two projections are checked separately
    hd = dev(_padded(h_o.astype(np.float32), rows), shape.dtype)
    y = D.empty(rows, shape.d_model, dtype=torch.float32)
    M.moe_expert_down(D.cfg, hd, off, D.weights, y, D.ws)
    torch.cuda.synchronize()
    assert_within_ulp(to_np(h)[:m], h_o, shape.dtype, "h")
    # y is an fp32 accumulation of exactly the same bf16 products
    assert_close_rms(to_np(y)[:m], y_o, 1e-4, "y")
    # both together: y also carries the GPU h's one-ulp differences, each
    # scaled by a down-projection weight, so the layer tolerance applies
    y2 = D.empty(rows, shape.d_model, dtype=torch.float32)
    M.moe_grouped_ffn(D.cfg, xp, off, D.weights, h, y2, D.ws)
    torch.cuda.synchronize()
    assert_close_rms(to_np(y2)[:m], y_o, rel_tol(shape.dtype), "y (grouped)")
    assert D.device_error() == M.MOE_OK


@pytest.mark.parametrize("name,N", FFN_CASES)
def test_expert_up_gather_matches_materialised_rows(name, N):
    """The up projection reading token rows through token_of_row equals the
    one reading the expert-sorted copy x_perm bit for bit (same products,
    same accumulation order), and so matches the oracle's h."""
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    idx, disp, x_perm = _oracle_dispatch_inputs(shape, inp)
    rows = shape.n_tokens * shape.top_k
    m = int(disp["offsets"][-1])
    off = torch.zeros(shape.n_experts + 1, dtype=torch.int32, device="cuda")
    ros = torch.zeros(rows, dtype=torch.int32, device="cuda")
    tor = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
    xp = D.empty(rows, shape.d_model)
    M.moe_dispatch_permute(D.cfg, dev(idx), D.t["x"], off, ros, tor, xp, None, D.ws)
    # the same grouping without the copy leaves x_perm alone
    tor2 = torch.full((rows,), -3, dtype=torch.int32, device="cuda")
    M.moe_dispatch_permute(D.cfg, dev(idx), None, off, ros, tor2, None, None, D.ws)
    h_ref = D.empty(rows, shape.d_ff)
    M.moe_expert_up(D.cfg, xp, off, D.weights, h_ref, D.ws)
    h = D.empty(rows, shape.d_ff)
    M.moe_expert_up_gather(D.cfg, D.t["x"], tor2, off, D.weights, h, D.ws)
    torch.cuda.synchronize()
    assert torch.equal(tor[:m], tor2[:m])
    assert np.array_equal(to_np(tor2)[:m], disp["token_of_row"])
    assert torch.equal(h[:m], h_ref[:m])
    h_o, _ = O.grouped_ffn(x_perm, disp["offsets"], inp.values, shape.expert,
                           shape.dtype)
    assert_within_ulp(to_np(h)[:m], h_o, shape.dtype, "h (gathered)")
    assert D.device_error() == M.MOE_OK


@pytest.mark.parametrize("name,N", [("qwen3_moe", 4096), ("deepseek_v3_block", 2048)])
def test_expert_up_gather_on_pairs(name, N):
    """Enough rows per expert for 256-row CTA-pair tiles: the gathered up
    projection still equals the one over x_perm bit for bit."""
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    idx, disp, _ = _oracle_dispatch_inputs(shape, inp)
    rows = shape.n_tokens * shape.top_k
    m = int(disp["offsets"][-1])
    off = torch.zeros(shape.n_experts + 1, dtype=torch.int32, device="cuda")
    ros = torch.zeros(rows, dtype=torch.int32, device="cuda")
    tor = torch.zeros(rows, dtype=torch.int32, device="cuda")
    xp = D.empty(rows, shape.d_model)
    M.moe_dispatch_permute(D.cfg, dev(idx), D.t["x"], off, ros, tor, xp, None, D.ws)
    h_ref = D.empty(rows, shape.d_ff)
    M.moe_expert_up(D.cfg, xp, off, D.weights, h_ref, D.ws)
    h = D.empty(rows, shape.d_ff)
    M.moe_expert_up_gather(D.cfg, D.t["x"], tor, off, D.weights, h, D.ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(tor)[:m], disp["token_of_row"])
    assert torch.equal(h[:m], h_ref[:m])
    assert D.device_error() == M.MOE_OK


def test_shared_ffn_parity():
    inp = inputs_for("deepseek_v3_block", 300)
    shape = inp.shape
    D = Device(inp)
    hs = D.empty(shape.n_tokens, shape.n_shared * shape.d_ff_shared)
    so = torch.empty(shape.n_tokens, shape.d_model, device="cuda")
    M.moe_shared_ffn(D.cfg, D.t["x"], D.weights, hs, so, D.ws)
    torch.cuda.synchronize()
    ref = O.shared_ffn(inp.values["x"], inp.values["ws1"], inp.values["ws3"],
                       inp.values["ws2"], shape.dtype)
    assert_close_rms(to_np(so), ref, rel_tol(shape.dtype), "shared")


# -------------------------------------------------------------- combine
@pytest.mark.parametrize("dtype", [W.DTYPE_F32, W.DTYPE_BF16])
@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("cf", [0.0, 1.0])
def test_combine_parity(dtype, shared, cf):
    N, E, k, d = 1000, 16, 4, 256
    rng = np.random.default_rng(5)
    idx = W.make_assignments(N, E, k, seed=8, zipf_s=1.0)
    disp = O.dispatch(idx, E, cf)
    m = int(disp["offsets"][-1])
    y = rng.standard_normal((N * k, d)).astype(np.float32)
    w = rng.random((N, k)).astype(np.float32)
    s = rng.standard_normal((N, d)).astype(np.float32) if shared else None
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d, dtype=dtype,
                 capacity_factor=cf)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    out = torch.empty(N, d, dtype=M.torch_dtype(dtype), device="cuda")
    M.moe_combine(cfg, dev(y), dev(disp["row_of_slot"].astype(np.int32)),
                  dev(w), dev(s) if shared else None, out, ws)
    torch.cuda.synchronize()
    exact = O.combine(y, disp["row_of_slot"], w, s)
    assert_output_close(to_np(out), exact, dtype, "out")
    # the fp32 sum itself is far inside the tolerance: a bf16 output is the
    # correctly rounded value except where the fp32 sum straddles a boundary
    if dtype == W.DTYPE_BF16:
        assert np.mean(to_np(out) != O.round_bf16(exact)) < 0.01


# ------------------------------------------- router GEMM + selection
ROUTER_CASES = [("toy_top2_fp32", None), ("capacity_top2_fp32", None),
                ("capacity_top2_bf16", None), ("deepseek_v3_block", 1000),
                ("qwen3_moe", 1000), ("decode_stream", None),
                # the CUDA-core router below 512 tokens: both CTA shapes,
                # ragged token counts
                ("toy_top2_fp32", 5), ("deepseek_v3_block", 37), ("qwen3_moe", 200),
                ("capacity_top2_fp32", 300), ("qwen3_moe", 511)]


@pytest.mark.parametrize("name,N", ROUTER_CASES)
def test_router_topk_parity(name, N):
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    n, E, k = shape.n_tokens, shape.n_experts, shape.top_k
    logits = torch.empty(n, E, device="cuda")
    idx = torch.empty(n, k, dtype=torch.int32, device="cuda")
    w = torch.empty(n, k, device="cuda")
    st, sts = D.stats()
    M.moe_router_topk(D.cfg, D.t["x"], D.weights, logits, idx, w, sts, D.ws)
    torch.cuda.synchronize()
    v = inp.values
    lg_o = O.router_logits(v["x"], v["w_router"], v.get("b_router"))
    lg = to_np(logits)
    tol_logit = 1e-4 if shape.dtype == W.DTYPE_BF16 else 1e-5
    assert np.max(np.abs(lg - lg_o)) <= tol_logit * max(1.0, np.abs(lg_o).max())
    keys = O.selection_keys(lg_o, shape.route, v.get("sel_bias"))
    margin = logit_margin(lg, lg_o)
    amb = ambiguous_tokens(keys, k, margin)
    i_o, w_o, p_o = O.route(lg_o, shape.route, k, v.get("sel_bias"))
    ig = to_np(idx)
    assert np.array_equal(ig[~amb], i_o[~amb])
    check_selection_valid(ig[amb], keys[amb], k, margin)
    assert np.allclose(to_np(w)[~amb], w_o[~amb], rtol=1e-3, atol=1e-5)
    # selection runs on exactly the logits the router wrote: on those, every
    # token's experts and slot order equal the oracle's, ties included
    i_g, w_g, _ = O.route(lg, shape.route, k, v.get("sel_bias"))
    assert np.array_equal(ig, i_g)
    assert np.allclose(to_np(w), w_g, rtol=1e-3, atol=1e-5)
    # without the logits output the selection is the same
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    M.moe_router_topk(D.cfg, D.t["x"], D.weights, None, idx2, w2, None, D.ws)
    torch.cuda.synchronize()
    assert torch.equal(idx2, idx) and torch.equal(w2, w)
    # the counts are those of the GPU's own selection
    cnt = np.bincount(ig.reshape(-1), minlength=E)
    assert np.array_equal(to_np(st["counts"]), cnt)
    if not amb.any():
        b_ref = O.balance_statistic(cnt, p_o, n, shape.balance_coef)
        assert abs(float(to_np(st["balance"])[0]) - b_ref) <= BALANCE_REL * abs(b_ref)


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
def test_router_ties_from_duplicated_experts(mode, dtype):
    """Experts with identical router rows (and selection bias) produce exactly
    equal keys: the lower expert index must win, on the tensor-core router
    (bf16) as on the CUDA-core one (fp32)."""
    E, k, d, N = 64, 6, 256, 333
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d, d_ff=64, dtype=dtype,
                 route=mode, sel_bias_range=0.1 if mode == 2 else 0.0)
    inp = W.make_inputs(shape)
    v = inp.values
    for src, dst in ((3, 40), (3, 17), (9, 10), (0, 63)):
        v["w_router"][dst] = v["w_router"][src]
        if "w_router" in inp.bits:
            inp.bits["w_router"][dst] = inp.bits["w_router"][src]
        if mode == 2:
            v["sel_bias"][dst] = v["sel_bias"][src]
    D = Device(inp)
    logits = torch.empty(N, E, device="cuda")
    idx = torch.empty(N, k, dtype=torch.int32, device="cuda")
    w = torch.empty(N, k, device="cuda")
    st, sts = D.stats()
    M.moe_router_topk(D.cfg, D.t["x"], D.weights, logits, idx, w, sts, D.ws)
    torch.cuda.synchronize()
    lg = to_np(logits)
    assert np.array_equal(lg[:, 40], lg[:, 3]) and np.array_equal(lg[:, 63], lg[:, 0])
    i_o, w_o, p_o = O.route(lg, mode, k, v.get("sel_bias"))
    assert np.array_equal(to_np(idx), i_o)
    assert np.allclose(to_np(w), w_o, rtol=1e-3, atol=1e-5)
    cnt = np.bincount(i_o.reshape(-1), minlength=E)
    assert np.array_equal(to_np(st["counts"]), cnt)
    b_ref = O.balance_statistic(cnt, p_o, N, shape.balance_coef)
    assert abs(float(to_np(st["balance"])[0]) - b_ref) <= BALANCE_REL * abs(b_ref)


# --------------------------------------------------------- whole layer
FORWARD_CASES = [("toy_top2_fp32", None), ("capacity_top2_fp32", None),
                 ("capacity_top2_bf16", None), ("deepseek_v3_block", 640),
                 ("qwen3_moe", 640), ("decode_stream", None)]


def _router_margin(D, ref_logits):
    """The near-tie margin of this layer's router: from the GPU router's
    logits (the same kernel moe_forward runs) against the oracle's."""
    shape = D.shape
    n, E, k = shape.n_tokens, shape.n_experts, shape.top_k
    logits = torch.zeros(n, E, device="cuda")
    idx = torch.zeros(n, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(n, k, device="cuda")
    M.moe_router_topk(D.cfg, D.t["x"], D.weights, logits, idx, w, None, D.ws)
    torch.cuda.synchronize()
    return logit_margin(to_np(logits), ref_logits)


def _forward(D, stats=True):
    shape = D.shape
    out = D.empty(shape.n_tokens, shape.d_model)
    st, sts = D.stats()
    M.moe_forward(D.cfg, D.t["x"], D.weights, out, sts if stats else None, D.ws)
    torch.cuda.synchronize()
    return out, st


@pytest.mark.parametrize("name,N", FORWARD_CASES)
def test_forward_parity(name, N):
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    out, st = _forward(D)
    ref = O.forward(shape, inp.values)
    margin = _router_margin(D, ref["logits"])
    keys = O.selection_keys(ref["logits"], shape.route, inp.values.get("sel_bias"))
    # a near-tie at the k-th key may swap one expert for another; with a
    # capacity that also moves later drops of the experts involved, so those
    # experts' tokens are left out of the exact comparison
    amb, swap = set_ambiguous_tokens(keys, shape.top_k, margin)
    keep = ~amb
    if shape.capacity_factor > 0 and swap:
        keep &= ~np.isin(ref["idx"], sorted(swap)).any(axis=1)
    if shape.capacity_factor > 0:
        others = np.array([e not in swap for e in range(shape.n_experts)])
        for n in ("kept", "dropped"):
            assert np.array_equal(to_np(st[n])[others], ref[n][others]), n
    assert keep.mean() > 0.9
    o = to_np(out)
    assert_output_close(o[keep], ref["out_exact"][keep], shape.dtype, name)
    cnt = to_np(st["counts"])
    assert cnt.sum() == shape.n_tokens * shape.top_k
    assert np.abs(cnt - ref["counts"]).sum() <= 2 * amb.sum()
    b = float(to_np(st["balance"])[0])
    if not amb.any():
        assert abs(b - ref["balance"]) <= BALANCE_REL * abs(ref["balance"])
    assert D.device_error() == M.MOE_OK


def test_forward_host_matches_forward():
    inp = inputs_for("capacity_top2_bf16", None)
    D = Device(inp)
    out, _ = _forward(D)
    shape = inp.shape
    xh = D.t["x"].cpu().pin_memory()
    oh = torch.empty(shape.n_tokens, shape.d_model, dtype=D.tdtype).pin_memory()
    M.moe_forward_host(D.cfg, xh, D.weights, oh, None, D.ws)
    torch.cuda.synchronize()
    assert torch.equal(oh, out.cpu())


@pytest.mark.parametrize("N", [12288 + 96, 8200])
def test_forward_host_pipelined_matches_forward(N):
    """Without a capacity, moe_forward_host splits the tokens into chunks and
    overlaps the host copies with the compute; the output and every
    statistic equal one moe_forward over all tokens, bit for bit (three
    chunks with a ragged tail; two chunks, the last under 4096 tokens)."""
    inp = inputs_for("qwen3_moe", N)
    D = Device(inp)
    shape = inp.shape
    out, st = _forward(D)
    xh = D.t["x"].cpu().pin_memory()
    oh = torch.full((shape.n_tokens, shape.d_model), 7.0, dtype=D.tdtype).pin_memory()
    st2, sts2 = D.stats()
    for _ in range(2):                                  # twice: the pipeline is reused
        M.moe_forward_host(D.cfg, xh, D.weights, oh, sts2, D.ws)
        torch.cuda.synchronize()
        assert torch.equal(oh, out.cpu())
        for name in ("counts", "kept", "dropped", "balance"):
            assert torch.equal(st2[name], st[name]), name
    assert D.device_error() == M.MOE_OK


def test_forward_timed_matches_forward():
    """The instrumented entry point makes the same launches: identical output
    and statistics, and its events bracket every stage in order."""
    inp = inputs_for("deepseek_v3_block", 300)
    D = Device(inp)
    a, sa = _forward(D)
    out = D.empty(D.shape.n_tokens, D.shape.d_model)
    st, sts = D.stats()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(M.MOE_FORWARD_EVENTS)]
    M.moe_forward_timed(D.cfg, D.t["x"], D.weights, out, sts, D.ws, evs)
    torch.cuda.synchronize()
    assert torch.equal(out, a)
    for name in ("counts", "kept", "dropped", "balance"):
        assert torch.equal(st[name], sa[name]), name
    gaps = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(evs) - 1)]
    assert all(g >= 0.0 for g in gaps) and sum(gaps) > 0.0
    with pytest.raises(ValueError):
        M.moe_forward_timed(D.cfg, D.t["x"], D.weights, out, sts, D.ws, evs[:3])


def test_forward_is_deterministic():
    inp = inputs_for("deepseek_v3_block", 256)
    D = Device(inp)
    a, sa = _forward(D)
    b, sb = _forward(D)
    assert torch.equal(a, b)
    assert torch.equal(sa["balance"], sb["balance"])


@pytest.mark.parametrize("name,N", [("deepseek_v3_block", 256), ("qwen3_moe", 4096)])
def test_forward_captures_into_a_cuda_graph(name, N):
    """No host synchronisation inside moe_forward (DSEEK failure modes): the
    whole layer is captured into a CUDA graph, and each replay gives the
    eager result bit for bit, outputs and statistics (4096 Qwen3-style
    tokens put the expert GEMMs on CTA pairs)."""
    inp = inputs_for(name, N)
    D = Device(inp)
    eager, se = _forward(D)
    out = D.empty(inp.shape.n_tokens, inp.shape.d_model)
    st, sts = D.stats()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            M.moe_forward(D.cfg, D.t["x"], D.weights, out, sts, D.ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        for key in ("counts", "kept", "dropped", "balance"):
            assert torch.equal(st[key], se[key]), key
    assert D.device_error() == M.MOE_OK


def test_forward_zero_tokens():
    inp = inputs_for("toy_top2_fp32", 0)
    D = Device(inp)
    out, st = _forward(D)
    assert out.numel() == 0
    assert (to_np(st["counts"]) == 0).all() and float(to_np(st["balance"])[0]) == 0.0


def _forward_vs_oracle(shape, what):
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, st = _forward(D)
    ref = O.forward(shape, inp.values)
    keys = O.selection_keys(ref["logits"], shape.route, inp.values.get("sel_bias"))
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, _router_margin(D, ref["logits"]))
    keep = ~amb
    assert keep.mean() > 0.9
    assert_output_close(to_np(out)[keep], ref["out_exact"][keep], shape.dtype, what)
    assert D.device_error() == M.MOE_OK
    return out, st, ref


def test_forward_256_experts():
    """The largest expert count: 256 SwiGLU experts, top-8 (selection with 8
    candidates per lane, 256 groups in the grouped GEMMs)."""
    shape = _cfg(n_tokens=700, n_experts=256, top_k=8, d_model=128, d_ff=64,
                 route=W.ROUTE_TOPK_SOFTMAX, dtype=W.DTYPE_BF16)
    _forward_vs_oracle(shape, "E=256")


@pytest.mark.parametrize("route", [0, 1, 2])
def test_forward_single_token(route):
    shape = _cfg(n_tokens=1, n_experts=16, top_k=4, d_model=128, d_ff=64, route=route,
                 dtype=W.DTYPE_BF16)
    if route == W.ROUTE_SIGMOID_BIAS:
        shape = shape.replace(sel_bias_range=0.1)
    _forward_vs_oracle(shape, "N=1")


def test_forward_capacity_drops_everything():
    """cf small enough that the capacity int(cf * (N // E)) is 0: every
    assignment is dropped and the layer output is exactly zero."""
    shape = _cfg(n_tokens=64, n_experts=8, top_k=2, d_model=64, d_ff=64,
                 dtype=W.DTYPE_BF16, capacity_factor=0.01)
    out, st, ref = _forward_vs_oracle(shape, "cap 0")
    assert torch.count_nonzero(out) == 0
    assert int(to_np(st["kept"]).sum()) == 0
    assert int(to_np(st["dropped"]).sum()) == 64 * 2


@pytest.mark.parametrize("E,k", [(1, 1), (4, 4)])
def test_forward_special_cases(E, k):
    """E = 1, k = 1 is the dense FFN; k = E with no capacity is the dense
    all-expert weighted sum -- both reach the same values as the oracle."""
    shape = _cfg(n_tokens=300, n_experts=E, top_k=k, d_model=64, d_ff=96)
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, _ = _forward(D)
    ref = O.forward(shape, inp.values)
    assert_output_close(to_np(out), ref["out_exact"], shape.dtype, "special")


@pytest.mark.parametrize("d", [48, 40, 272])
def test_forward_bf16_row_widths(d):
    """bf16 layers whose rows are not a multiple of the combine's 32-byte
    pieces (40: 16-byte path) or hold only a few of them (48, 272: several
    tokens per CTA) still match the oracle."""
    shape = _cfg(n_tokens=300, n_experts=8, top_k=2, d_model=d, d_ff=64,
                 dtype=W.DTYPE_BF16)
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, _ = _forward(D)
    ref = O.forward(shape, inp.values)
    assert_output_close(to_np(out), ref["out_exact"], shape.dtype, "row widths")


@pytest.mark.parametrize("expert,N,d,F", [(W.EXPERT_SILU_MLP, 300, 64, 72),
                                          (W.EXPERT_SWIGLU, 600, 72, 64)])
def test_forward_bf16_k_not_whole_blocks(expert, N, d, F):
    """Tensor-core GEMMs whose reduction length is not a whole number of
    64-wide k-blocks: the down projection (K = F = 72) and the router GEMM
    (K = d = 72, 600 tokens) read the right B columns in their last block."""
    shape = _cfg(n_tokens=N, n_experts=8, top_k=2, d_model=d, d_ff=F, expert=expert,
                 has_bias=expert == W.EXPERT_SILU_MLP, dtype=W.DTYPE_BF16)
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, _ = _forward(D)
    ref = O.forward(shape, inp.values)
    keys = O.selection_keys(ref["logits"], shape.route, None)
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, _router_margin(D, ref["logits"]))
    keep = ~amb
    assert keep.mean() > 0.9
    assert_output_close(to_np(out)[keep], ref["out_exact"][keep], shape.dtype, "k tail")


# -------------------------------------------- full-size sampled checks
@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen3_moe", "deepseek_v3_block"])
def test_forward_full_size_sampled(name):
    inp = inputs_for(name, None)
    shape = inp.shape
    D = Device(inp)
    out, st = _forward(D)
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([rng.choice(shape.n_tokens, 48, replace=False),
                                       [0, shape.n_tokens - 1]]))
    ref = O.forward_tokens(shape, inp.values, tokens)
    keys = O.selection_keys(ref["logits"], shape.route, inp.values.get("sel_bias"))
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, 4e-4)   # logits agree to 1e-4
    o = to_np(out)[tokens]
    assert_output_close(o[~amb], ref["out_exact"][~amb], shape.dtype, name)
    cnt = to_np(st["counts"])
    assert cnt.sum() == shape.n_tokens * shape.top_k
    assert D.device_error() == M.MOE_OK


# ------------------------------------------- between steps: bias update
@pytest.mark.parametrize("E", [1, 3, 8, 64, 128, 256])
@pytest.mark.parametrize("gamma", [1e-3, 0.37])
def test_selection_bias_update_bit_exact(E, gamma):
    rng = np.random.default_rng(1000 + E)
    counts = rng.integers(0, 50, E).astype(np.int32)
    if E >= 3:
        counts[:3] = 0                     # idle experts
        counts[-1] = counts.sum() // E     # may sit exactly at the mean
    bias = rng.standard_normal(E).astype(np.float32)
    bias[0] = -0.0
    shape = _cfg(n_experts=E, top_k=1)
    cfg = M.make_config(shape)
    dc = torch.from_numpy(counts).cuda()
    db = torch.from_numpy(bias.copy()).cuda()
    cv = torch.full((1,), -1.0, device="cuda")
    for step in range(2):                  # two updates in a row
        M.moe_update_selection_bias(cfg, dc, db, gamma, cv)
        bias = O.selection_bias_update(bias, counts, gamma)
        torch.cuda.synchronize()
        got = db.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), bias.view(np.uint32)), step
        ref_cv = O.load_cv(counts)
        assert abs(float(to_np(cv)[0]) - ref_cv) <= 1e-6 * max(ref_cv, 1e-30)


def test_selection_bias_update_degenerate_loads():
    E = 16
    cfg = M.make_config(_cfg(n_experts=E, top_k=1))
    bias = torch.linspace(-1, 1, E, device="cuda")
    before = bias.clone()
    cv = torch.full((1,), -1.0, device="cuda")
    # nothing routed: every expert sits at the mean, CV 0
    M.moe_update_selection_bias(cfg, torch.zeros(E, dtype=torch.int32, device="cuda"),
                                bias, 0.5, cv)
    torch.cuda.synchronize()
    assert torch.equal(bias, before) and float(cv[0]) == 0.0
    # perfectly balanced: same
    M.moe_update_selection_bias(cfg, torch.full((E,), 7, dtype=torch.int32, device="cuda"),
                                bias, 0.5, cv)
    torch.cuda.synchronize()
    assert torch.equal(bias, before) and float(cv[0]) == 0.0
    # everything on one expert: CV = sqrt(E - 1); only load_cv requested
    c = torch.zeros(E, dtype=torch.int32, device="cuda")
    c[5] = 1000
    M.moe_update_selection_bias(cfg, c, None, 0.5, cv)
    torch.cuda.synchronize()
    assert abs(float(cv[0]) - (E - 1) ** 0.5) <= 1e-6 * (E - 1) ** 0.5


def test_selection_bias_update_from_forward_counts():
    """The counts a sigmoid-bias forward reports feed the update directly."""
    inp = inputs_for("deepseek_v3_block", 256)
    D = Device(inp)
    _, st = _forward(D)
    shape = inp.shape
    cfg = M.make_config(shape)
    bias0 = inp.values["sel_bias"].astype(np.float32)
    db = torch.from_numpy(bias0.copy()).cuda()
    M.moe_update_selection_bias(cfg, st["counts"], db, 1e-3, None)
    torch.cuda.synchronize()
    ref = O.selection_bias_update(bias0, to_np(st["counts"]), 1e-3)
    assert np.array_equal(db.cpu().numpy().view(np.uint32), ref.view(np.uint32))
