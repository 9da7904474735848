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


@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (256, 8)])
@pytest.mark.parametrize("spread", [1e-3, 1.0])
def test_route_sigmoid_large_bias_bit_exact(E, k, spread):
    """Selection biases of magnitude ~10^3 ("DeepSeek 5.7", s.2 puts no bound
    on the balancing bias): one ulp of a key s + b is then 2^-14..2^-13, far
    above the error of the fast fp32 sigmoid, so the candidates that get the
    exact (double) sigmoid must be chosen relative to the key's magnitude.
    Biases sit on a few shared values, some straddling the binade boundary
    at 1024, and narrow logits (spread 1e-3) put many keys within an ulp of
    one another: exact ties to the lower index and one-ulp near-ties
    everywhere.  idx must equal the all-double definition bit for bit."""
    N = 1000
    rng = np.random.default_rng(E * 10 + k + int(spread * 7))
    levels = np.array([1023.75, 1023.9375, 1000.0, 1000.0, 2047.5, -999.0],
                      np.float32)
    bias = levels[rng.integers(0, len(levels), E)]
    # k + 2 experts (all of them for small E) share the top level, whose keys
    # s + 2047.5 straddle the binade boundary at 2048 (ulps 2^-12 / 2^-11)
    bias[rng.permutation(E)[:min(E, k + 2)]] = np.float32(2047.5)
    logits = (spread * rng.standard_normal((N, E))).astype(np.float32)
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, route=W.ROUTE_SIGMOID_BIAS)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    idx = torch.full((N, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((N, k), dtype=torch.float32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    bal = torch.zeros(1, dtype=torch.float32, device="cuda")
    M.moe_route_logits(cfg, dev(logits), dev(bias), idx, w,
                       M.make_stats(counts=counts, balance=bal), ws)
    torch.cuda.synchronize()
    i_o, w_o, p_o = O.route(logits, W.ROUTE_SIGMOID_BIAS, k, bias)
    keys = O.selection_keys(logits, W.ROUTE_SIGMOID_BIAS, bias)
    # the case is what it claims: many exact ties at the k-th key
    kth = -np.sort(-keys, axis=1)[:, k - 1]
    assert ((keys == kth[:, None]).sum(axis=1) > 1).mean() > (0.2 if spread < 0.1 else 0.0)
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


@pytest.mark.parametrize("N,E,k,cf,zipf", DISPATCH_CASES)
def test_check_grouping_accepts_every_dispatch(N, E, k, cf, zipf):
    """The device-side consistency check passes on every grouping the
    dispatch writes (capacity drops, N < E, k = E, E = 1, many empty
    experts)."""
    idx = W.make_assignments(N, E, k, seed=N + 2 * E + k, zipf_s=zipf)
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, capacity_factor=cf)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    di = dev(idx)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    ros = torch.zeros(N * k, dtype=torch.int32, device="cuda")
    tor = torch.zeros(N * k, dtype=torch.int32, device="cuda")
    M.moe_dispatch_permute(cfg, di, None, offsets, ros, tor, None, None, ws)
    for _ in range(2):                      # its counters are left zero: twice in a row
        M.moe_check_grouping(cfg, di, offsets, ros, tor, ws)
        assert M.moe_read_device_error(ws) == M.MOE_OK


def _planted_groupings(idx, offsets, ros, tor, k):
    """Inconsistent groupings, each one mistake away from a valid one, every
    index still inside its buffer (so the check reads nothing out of range)."""
    kept = np.nonzero(ros >= 0)[0]
    a, b = kept[0], kept[len(kept) // 2]
    out = []
    r = ros.copy(); r[a], r[b] = r[b], r[a]
    out.append(("rows swapped", idx, offsets, r, tor))
    r = ros.copy(); r[b] = -1
    out.append(("kept slot marked dropped", idx, offsets, r, tor))
    t = tor.copy(); t[ros[b]] = (t[ros[b]] + 1) % (idx.shape[0])
    out.append(("token_of_row wrong", idx, offsets, ros, t))
    o = offsets.copy(); o[1], o[2] = o[2], o[1]
    out.append(("offsets decrease", idx, o, ros, tor))
    i = idx.copy(); i[0, 1] = i[0, 0]
    out.append(("duplicate expert in a token", i, offsets, ros, tor))
    return out


def test_check_grouping_flags_planted_inconsistencies():
    N, E, k = 1000, 16, 4
    idx = W.make_assignments(N, E, k, seed=9, zipf_s=1.0)
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k)
    cfg = M.make_config(shape)
    ws = M.MoEWorkspace(cfg, forward=False)
    disp = O.dispatch(idx, E, 0.0)
    base = (idx.astype(np.int32), disp["offsets"].astype(np.int32),
            disp["row_of_slot"].astype(np.int32), disp["token_of_row"].astype(np.int32))
    M.moe_check_grouping(cfg, *(dev(a) for a in base), ws)
    assert M.moe_read_device_error(ws) == M.MOE_OK       # the oracle's grouping passes
    tor_full = np.zeros(N * k, np.int32)
    tor_full[:len(base[3])] = base[3]
    for what, i, o, r, t in _planted_groupings(base[0], base[1], base[2], tor_full, k):
        M.moe_check_grouping(cfg, dev(i), dev(o), dev(r), dev(t), ws)
        assert M.moe_read_device_error(ws) == M.MOE_ERR_DEVICE_CHECK, what
    # and the check's own counters were left clean
    M.moe_check_grouping(cfg, *(dev(a) for a in (base[0], base[1], base[2], tor_full)), ws)
    assert M.moe_read_device_error(ws) == M.MOE_OK


@pytest.mark.parametrize("dtype", [W.DTYPE_BF16, W.DTYPE_F32])
def test_grouped_gemm_refuses_inconsistent_offsets(dtype):
    """Offsets that decrease, or end past the grouped buffer, set the error
    word and the grouped GEMM writes nothing (tensor-core and CUDA-core)."""
    N, E, k, d, F = 256, 8, 2, 64, 64
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d, d_ff=F, dtype=dtype)
    inp = W.make_inputs(shape)
    D = Device(inp)
    xp = D.empty(N * k, d)
    good = np.linspace(0, N * k, E + 1).astype(np.int32)
    for what, off in (("decreasing", np.r_[good[:3], good[2] - 5, good[4:]]),
                      ("past the buffer", np.r_[good[:-1], N * k + 64])):
        assert off.min() >= 0 and len(off) == E + 1, what
        h = torch.full((N * k, F), 3.0, dtype=D.tdtype, device="cuda")
        M.moe_expert_up(D.cfg, xp, dev(off.astype(np.int32)), D.weights, h, D.ws)
        torch.cuda.synchronize()
        assert D.device_error() == M.MOE_ERR_DEVICE_CHECK, what
        assert bool((h == 3.0).all()), what


# ---------------------------------------------------------- expert FFNs
FFN_CASES = [("toy_top2_fp32", 64), ("capacity_top2_fp32", 700),
             ("capacity_top2_bf16", 700), ("deepseek_v3_block", 300),
             ("qwen3_moe", 200),
             # enough rows per expert for CTA pairs, with short group tails
             # left to the single-CTA pass
             ("deepseek_v3_block", 1536),
             # a few rows per expert: the swapped-operand kernel (weights on
             # the MMA's M side), SwiGLU and SiLU + bias
             ("decode_stream", None), ("capacity_top2_bf16", 48)]


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
    # the counts are those of the GPU's own selection, and the balance
    # statistic is the oracle's on the GPU's own logits and counts (near-ties
    # or not)
    cnt = np.bincount(ig.reshape(-1), minlength=E)
    assert np.array_equal(to_np(st["counts"]), cnt)
    _, _, p_g = O.route(lg, shape.route, k, v.get("sel_bias"))
    b_ref = O.balance_statistic(cnt, p_g, n, shape.balance_coef)
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
                 ("qwen3_moe", 640), ("decode_stream", None),
                 # a few rows per expert, biases and a capacity that drops:
                 # the swapped-operand up and compact down projections
                 ("capacity_top2_bf16", 48), ("deepseek_v3_block", 96)]


def _gpu_logits(D):
    """The router logits moe_forward works from: the same router kernels
    (chosen by the token count), written out by moe_router_topk."""
    shape = D.shape
    n, E, k = shape.n_tokens, shape.n_experts, shape.top_k
    logits = torch.zeros(n, E, device="cuda")
    idx = torch.zeros(n, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(n, k, device="cuda")
    M.moe_router_topk(D.cfg, D.t["x"], D.weights, logits, idx, w, None, D.ws)
    torch.cuda.synchronize()
    return to_np(logits)


def _router_margin(D, ref_logits):
    """The near-tie margin of this layer's router: from the GPU router's
    logits (the same kernel moe_forward runs) against the oracle's."""
    return logit_margin(_gpu_logits(D), ref_logits)


def _check_forward_statistics(D, st, lg_gpu, values):
    """The forward's selection counts and balance statistic against the
    oracle's selection and statistic computed on the GPU's own logits: the
    counts bit-exact, the statistic within 1e-4 relative, whatever near-ties
    the layer holds.  With a capacity, kept/dropped must then equal the
    oracle's grouping of that same selection."""
    shape = D.shape
    i_g, _, p_g = O.route(lg_gpu, shape.route, shape.top_k, values.get("sel_bias"))
    cnt = np.bincount(i_g.reshape(-1), minlength=shape.n_experts)
    assert np.array_equal(to_np(st["counts"]), cnt)
    b_ref = O.balance_statistic(cnt, p_g, shape.n_tokens, shape.balance_coef)
    assert abs(float(to_np(st["balance"])[0]) - b_ref) <= BALANCE_REL * abs(b_ref)
    disp = O.dispatch(i_g, shape.n_experts, float(np.float32(shape.capacity_factor)))
    for name in ("kept", "dropped"):
        assert np.array_equal(to_np(st[name]), disp[name]), name


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
    lg_gpu = _gpu_logits(D)
    margin = logit_margin(lg_gpu, ref["logits"])
    _check_forward_statistics(D, st, lg_gpu, inp.values)
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
    assert D.device_error() == M.MOE_OK


def test_forward_combine_register_path():
    """A token whose k compact rows do not fit a bulk-copy stage (d = 2304,
    top-8: 37.4 KB per token) takes the register-fed combine; the whole
    output against the oracle."""
    shape = W.WORKLOADS["qwen3_moe"].replace(name="wide_d", n_tokens=512, n_experts=16,
                                             d_model=2304)
    assert shape.top_k * shape.d_model * 2 + shape.top_k * shape.d_model // 32 > 36 * 1024
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, st = _forward(D)
    ref = O.forward(shape, inp.values)
    lg_gpu = _gpu_logits(D)
    keys = O.selection_keys(ref["logits"], shape.route, inp.values.get("sel_bias"))
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, logit_margin(lg_gpu, ref["logits"]))
    assert (~amb).mean() > 0.9
    assert_output_close(to_np(out)[~amb], ref["out_exact"][~amb], shape.dtype, "wide_d")
    assert D.device_error() == M.MOE_OK


@pytest.mark.parametrize("name,N", [("qwen3_moe", 4096), ("deepseek_v3_block", 4096)])
def test_forward_whole_output_large(name, N):
    """Every output of a 4096-token layer against the oracle: the expert
    GEMMs run on CTA pairs with the compact, weighted, slot-ordered down
    projection, and the selection sums its statistic over 32-token CTAs
    (the path of the full-size layers)."""
    inp = inputs_for(name, N)
    shape = inp.shape
    D = Device(inp)
    out, st = _forward(D)
    ref = O.forward(shape, inp.values)
    lg_gpu = _gpu_logits(D)
    _check_forward_statistics(D, st, lg_gpu, inp.values)
    keys = O.selection_keys(ref["logits"], shape.route, inp.values.get("sel_bias"))
    amb, _ = set_ambiguous_tokens(keys, shape.top_k, logit_margin(lg_gpu, ref["logits"]))
    assert (~amb).mean() > 0.9
    assert_output_close(to_np(out)[~amb], ref["out_exact"][~amb], shape.dtype, name)
    # near-tie tokens: the GPU's own selection, weights and output from the
    # oracle's experts on those same choices
    if amb.any():
        tok = np.nonzero(amb)[0]
        i_g, w_g, _ = O.route(lg_gpu[tok], shape.route, shape.top_k,
                              inp.values.get("sel_bias"))
        v = inp.values
        exact = np.zeros((len(tok), shape.d_model))
        for i, t in enumerate(tok):
            for j in range(shape.top_k):
                e = int(i_g[i, j])
                _, y = O.expert_ffn(v["x"][t:t + 1], v["w1"][e], v["w2"][e], shape.expert,
                                    shape.dtype, w3=v["w3"][e])
                exact[i] += w_g[i, j] * y[0]
        if shape.n_shared > 0:
            exact += O.round_f32(O.shared_ffn(v["x"][tok], v["ws1"], v["ws3"], v["ws2"],
                                              shape.dtype))
        rms = float(np.sqrt(np.mean(ref["out_exact"] ** 2)))
        err = np.abs(to_np(out)[tok] - exact)
        assert (err <= 2e-2 * rms + np.abs(exact) * 2.0 ** -8).all()
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


@pytest.mark.parametrize("N", [16384, 12288 + 96, 8200])
def test_forward_host_pipelined_matches_forward(N):
    """Without a capacity, moe_forward_host splits the tokens into chunks and
    overlaps the host copies with the compute; the output and every
    statistic equal one moe_forward over all tokens, bit for bit (four
    chunks in the proportions 3:5:5:3 over the whole layer; three in 3:5:3;
    two equal chunks with a ragged tail)."""
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
    # counts and balance statistic of the whole layer (32-token selection
    # CTAs) against the oracle's on the GPU's own logits of every token
    _check_forward_statistics(D, st, _gpu_logits(D), inp.values)
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


# ------------------------------------------- grouping with a per-expert room
@pytest.mark.parametrize("N,E,k,cf,zipf", DISPATCH_CASES)
def test_dispatch_room_bit_exact(N, E, k, cf, zipf):
    """Grouping with one capacity per expert (room [E]: zero, negative, below
    and above the expert's load) equals the oracle's grouping with those
    capacities, bit for bit; a room of the scalar capacity everywhere equals
    moe_dispatch_permute with capacity_factor."""
    d = 32
    idx = W.make_assignments(N, E, k, seed=N + E + k + 1, zipf_s=zipf)
    x = np.random.default_rng(N + 1).standard_normal((N, d)).astype(np.float32)
    shape = _cfg(n_tokens=N, n_experts=E, top_k=k, d_model=d, capacity_factor=cf,
                 dtype=W.DTYPE_BF16)
    cfg = M.make_config(shape)
    cfg_nocap = M.make_config(shape.replace(capacity_factor=0.0))
    ws = M.MoEWorkspace(cfg, forward=False)
    xd, di = dev(x, W.DTYPE_BF16), dev(idx)
    load = np.bincount(idx.reshape(-1), minlength=E)
    rng = np.random.default_rng(E + k)
    rooms = [rng.integers(-3, max(2, int(load.max()) + 3), E).astype(np.int32),
             np.zeros(E, np.int32), (load // 2).astype(np.int32)]
    cap = O.capacity(float(np.float32(cf)), N, E)
    if cap is not None:
        rooms.append(np.full(E, cap, np.int32))

    def run(room):
        o = dict(offsets=torch.full((E + 1,), -5, dtype=torch.int32, device="cuda"),
                 ros=torch.full((N * k,), -5, dtype=torch.int32, device="cuda"),
                 tor=torch.full((N * k,), -5, dtype=torch.int32, device="cuda"),
                 xp=torch.zeros((N * k, d), dtype=torch.bfloat16, device="cuda"))
        st = {n: torch.full((E,), -5, dtype=torch.int32, device="cuda")
              for n in ("counts", "kept", "dropped")}
        if room is None:
            M.moe_dispatch_permute(cfg, di, xd, o["offsets"], o["ros"], o["tor"], o["xp"],
                                   M.make_stats(**st), ws)
        else:
            M.moe_dispatch_permute_room(cfg, di, xd, dev(room), o["offsets"], o["ros"],
                                        o["tor"], o["xp"], M.make_stats(**st), ws)
        # (a per-expert room may exceed the config's capacity: the check
        # runs on a config without one)
        M.moe_check_grouping(cfg_nocap, di, o["offsets"], o["ros"], o["tor"], ws)
        torch.cuda.synchronize()
        assert M.moe_read_device_error(ws) == M.MOE_OK
        o.update(st)
        return o

    for room in rooms:
        got = run(room)
        res = O.dispatch(idx, E, expert_capacity=room)
        m = int(res["offsets"][-1])
        assert np.array_equal(to_np(got["offsets"]), res["offsets"])
        assert np.array_equal(to_np(got["ros"]), res["row_of_slot"])
        assert np.array_equal(to_np(got["tor"])[:m], res["token_of_row"])
        for n in ("counts", "kept", "dropped"):
            assert np.array_equal(to_np(got[n]), res[n]), n
        ref = xd[torch.from_numpy(res["token_of_row"]).cuda()] if m else got["xp"][:0]
        assert torch.equal(got["xp"][:m].view(torch.int16), ref.view(torch.int16))
    if cap is not None:
        a, b = run(None), run(rooms[-1])
        for key in a:
            assert torch.equal(a[key], b[key]), key


# --------------------------------------------- the pages' worked example
@pytest.mark.parametrize("k", [2, 4])
def test_forward_worked_example(k):
    """"DeepSeek 5.7", Worked example, at its own sizes: B = 2, T = 4,
    d = 16, four routed SwiGLU experts, top-2 (and top-4: every expert),
    one shared expert, sigmoid routing with a selection bias.  The output is
    [2, 4, 16] (one row per token), each token has exactly k routed
    assignments, and the layer matches the oracle on the GPU's own routing;
    with k = E it is the dense all-expert sum with weights s_e / sum s."""
    shape = W.MoEShape(name="worked", n_tokens=8, d_model=16, n_experts=4, top_k=k, d_ff=64,
                       expert=W.EXPERT_SWIGLU, route=W.ROUTE_SIGMOID_BIAS,
                       dtype=W.DTYPE_BF16, sel_bias_range=0.1, n_shared=1, d_ff_shared=32,
                       seed=5)
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, st = _forward(D)
    assert tuple(out.reshape(2, 4, 16).shape) == (2, 4, 16)
    assert np.array_equal(to_np(st["counts"]).sum(), 8 * k)
    v = inp.values
    lg = _gpu_logits(D)
    i_g, w_g, _ = O.route(lg, shape.route, k, v["sel_bias"])
    assert all(len(set(r)) == k for r in i_g.tolist())
    exact = np.zeros((8, 16))
    for t in range(8):
        for j in range(k):
            e = int(i_g[t, j])
            _, y = O.expert_ffn(v["x"][t:t + 1], v["w1"][e], v["w2"][e], shape.expert,
                                shape.dtype, w3=v["w3"][e])
            exact[t] += w_g[t, j] * y[0]
    exact += O.round_f32(O.shared_ffn(v["x"], v["ws1"], v["ws3"], v["ws2"], shape.dtype))
    assert_output_close(to_np(out), exact, shape.dtype, "worked example")
    if k == shape.n_experts:
        # dense: every expert, weight sigmoid(l_e) / sum over all experts
        s = O.sigmoid_f32(lg).astype(np.float64)
        dense = np.zeros((8, 16))
        for e in range(4):
            _, y = O.expert_ffn(v["x"], v["w1"][e], v["w2"][e], shape.expert, shape.dtype,
                                w3=v["w3"][e])
            dense += (s[:, e] / s.sum(axis=1))[:, None] * y
        dense += O.round_f32(O.shared_ffn(v["x"], v["ws1"], v["ws3"], v["ws2"], shape.dtype))
        assert_output_close(to_np(out), dense, shape.dtype, "dense all-expert sum")
    _check_forward_statistics(D, st, lg, v)
    assert D.device_error() == M.MOE_OK


@pytest.mark.parametrize("d", [64, 96, 160])
def test_forward_swapped_gemm_feature_tail(d):
    """A few rows per expert (the swapped-operand GEMMs) with d_model not a
    multiple of the 128 features a weight tile holds: the tile's last lane
    quadrants lie past d and must write nothing, neither values nor the
    compact output's block exponents (which would land on the next row's).
    Every output against the oracle on the GPU's own routing."""
    shape = _cfg(n_tokens=40, n_experts=16, top_k=2, d_model=d, d_ff=64,
                 route=W.ROUTE_TOPK_SOFTMAX, dtype=W.DTYPE_BF16)
    inp = W.make_inputs(shape)
    D = Device(inp)
    out, st = _forward(D)
    v = inp.values
    lg = _gpu_logits(D)
    i_g, w_g, _ = O.route(lg, shape.route, shape.top_k)
    exact = np.zeros((shape.n_tokens, d))
    for t in range(shape.n_tokens):
        for j in range(shape.top_k):
            e = int(i_g[t, j])
            _, y = O.expert_ffn(v["x"][t:t + 1], v["w1"][e], v["w2"][e], shape.expert,
                                shape.dtype, w3=v["w3"][e])
            exact[t] += w_g[t, j] * y[0]
    assert_output_close(to_np(out), exact, shape.dtype, f"d={d}")
    _check_forward_statistics(D, st, lg, v)
    assert D.device_error() == M.MOE_OK
