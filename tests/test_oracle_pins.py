"""Pins for the CPU oracle: checks against what the pages print, closed
forms, library routines and brute force -- never against the oracle itself.

Each test names the page section it pins.  The float64 library references
(torch.nn.functional in float64, torch.softmax, index_add_) are independent
of the oracle's numpy code paths.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

from oracle import moe_oracle as O
from routing_dispatch_expert_05_b300 import workloads as W
from tests.conftest import read_golden


def _golden_dict(name):
    out = {}
    for row in read_golden(name):
        out.setdefault(row[0], []).append(row[1:])
    return out


# ---------------------------------------------------------------- Out[9]
def test_param_count_matches_printed_out9():
    g = _golden_dict("expert_params.txt")
    d, f = int(g["d_model"][0][0]), int(g["d_ff"][0][0])
    n_exp = int(g["num_experts"][0][0])
    per = O.expert_param_count(d, f, bias=True)
    assert per == int(g["params_per_expert"][0][0])
    assert per * n_exp == int(g["total_params"][0][0])


def test_generated_capacity_workload_has_printed_param_count():
    """The capacity workload's tensors have the page's per-expert shapes."""
    shape = W.WORKLOADS["capacity_top2_fp32"]
    inp = W.make_inputs(shape, n_tokens=8)
    per_expert = sum(inp.values[n][0].size for n in ("w1", "b1", "w2", "b2"))
    g = _golden_dict("expert_params.txt")
    assert per_expert == int(g["params_per_expert"][0][0])
    total = sum(inp.values[n].size for n in ("w1", "b1", "w2", "b2"))
    assert total == int(g["total_params"][0][0])


# ---------------------------------------------------------------- Out[12]
def _table_assignments(seed=7):
    g = _golden_dict("capacity_table.txt")
    counts = [int(r[1]) for r in g["expert"]]
    idx = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    np.random.default_rng(seed).shuffle(idx)
    return g, counts, idx.reshape(-1, 1).astype(np.int32)


def test_capacity_truncates_tokens_per_expert_first():
    """EXPERT In[10] (reading R1): capacity = int(cf * (N // E)).  The
    tokens per expert are an integer division before the factor applies, so
    a ragged N gives a smaller capacity than int(cf * N / E) would."""
    assert O.capacity(2.0, 11, 4) == 4          # int(2.0 * 2), not int(5.5) = 5
    assert O.capacity(1.25, 7, 2) == 3          # int(1.25 * 3), not int(4.375) = 4
    assert O.capacity(0.5, 3, 4) == 0           # fewer tokens than experts: nothing kept
    assert O.capacity(0.0, 100, 4) is None and O.capacity(-1.0, 100, 4) is None
    d = O.dispatch(np.array([[0], [0], [0], [0], [0], [1], [1]]), 2, 1.25)
    assert d["kept"].tolist() == [3, 2] and d["dropped"].tolist() == [2, 0]


def test_dispatch_with_per_expert_capacities():
    """EXPERT In[10]'s token-order rule with one capacity per expert (a
    shard's remaining room): caps (1, 2) keep the first assignment to
    expert 0 and the first two to expert 1."""
    idx = np.array([[0], [0], [1], [0], [1], [1]])
    d = O.dispatch(idx, 2, expert_capacity=[1, 2])
    assert d["kept"].tolist() == [1, 2] and d["dropped"].tolist() == [2, 1]
    assert d["row_of_slot"].tolist() == [0, -1, 1, -1, 2, -1]
    assert d["token_of_row"].tolist() == [0, 2, 4]
    # zero room drops everything; the scalar rule is the broadcast case
    assert O.dispatch(idx, 2, expert_capacity=[0, 0])["kept"].tolist() == [0, 0]
    rng = np.random.default_rng(3)
    for cf in (0.5, 1.0, 1.25):
        idx = np.stack([rng.permutation(6)[:2] for _ in range(40)])
        a = O.dispatch(idx, 6, cf)
        b = O.dispatch(idx, 6, expert_capacity=[a["capacity"]] * 6)
        for key in ("kept", "dropped", "offsets", "row_of_slot", "token_of_row"):
            assert np.array_equal(a[key], b[key]), key


def test_capacity_table_out12():
    g, counts, idx = _table_assignments()
    n_tok = int(g["num_tokens"][0][0])
    n_exp = int(g["num_experts"][0][0])
    cf = float(g["capacity_factor"][0][0])
    assert idx.shape[0] == n_tok
    assert n_tok // n_exp == int(g["base_capacity"][0][0])
    assert O.capacity(cf, n_tok, n_exp) == int(g["capacity"][0][0])
    res = O.dispatch(idx, n_exp, cf)
    for e, row in enumerate(g["expert"]):
        assert int(row[0]) == e
        assert res["counts"][e] == int(row[1])
        assert res["kept"][e] == int(row[2])
        assert res["dropped"][e] == int(row[3])
    rate = 100.0 * res["dropped"].sum() / n_tok
    assert round(rate, 1) == float(g["total_drop_rate_percent"][0][0])


def test_drop_rate_sweep_out15():
    g = _golden_dict("drop_sweep.txt")
    _, _, idx = _table_assignments(seed=11)
    cfs = [float(c) for c in g["capacity_factors"][0]]
    rates = {}
    for cf in cfs:
        res = O.dispatch(idx, 8, cf)
        rates[cf] = 100.0 * res["dropped"].sum() / idx.shape[0]
    for cf_s, pct in g["approx_drop_percent_at"]:
        assert round(rates[float(cf_s)]) == int(pct)
    # more capacity never drops more
    vals = [rates[c] for c in cfs]
    assert all(a >= b for a, b in zip(vals, vals[1:]))


# ------------------------------------------------ dispatch: brute force
def _kept_by_definition(idx, cap):
    """Slot (t, j) is kept iff fewer than cap earlier tokens chose the same
    expert (the token-order capacity rule, stated as a count)."""
    n, k = idx.shape
    kept = np.zeros(n * k, bool)
    for t in range(n):
        for j in range(k):
            e = idx[t, j]
            earlier = sum(1 for u in range(t) if e in idx[u])
            kept[t * k + j] = cap is None or earlier < cap
    return kept


@pytest.mark.parametrize("n_tok,n_exp,k,cf", [
    (4, 2, 1, 0.5), (4, 2, 1, 1.0), (4, 3, 2, 1.0), (3, 3, 2, 1.0),
    (4, 3, 1, 2.0), (2, 4, 2, 1.0), (4, 2, 2, 0.0)])
def test_dispatch_all_assignments_brute_force(n_tok, n_exp, k, cf):
    cap = O.capacity(cf, n_tok, n_exp)
    per_token = list(itertools.permutations(range(n_exp), k))
    for combo in itertools.product(per_token, repeat=n_tok):
        idx = np.array(combo, np.int32).reshape(n_tok, k)
        res = O.dispatch(idx, n_exp, cf)
        kept = _kept_by_definition(idx, cap)
        assert np.array_equal(res["row_of_slot"] >= 0, kept)
        # rows of kept slots: sorted by (expert, token) -> 0..M-1
        slots = [s for s in range(n_tok * k) if kept[s]]
        order = sorted(slots, key=lambda s: (idx.reshape(-1)[s], s // k))
        expect_rows = np.full(n_tok * k, -1)
        for r, s in enumerate(order):
            expect_rows[s] = r
        assert np.array_equal(res["row_of_slot"], expect_rows)
        assert res["counts"].sum() == n_tok * k
        assert res["kept"].sum() == n_tok * k - res["dropped"].sum()
        if cap is not None:
            assert (res["kept"] <= cap).all()
        assert np.array_equal(
            res["token_of_row"], np.array([s // k for s in order], np.int64))


def test_dispatch_fewer_tokens_than_experts_drops_all_under_capacity():
    idx = np.array([[0, 1], [2, 0]], np.int32)
    res = O.dispatch(idx, 5, 1.25)           # cap = int(1.25 * (2 // 5)) = 0
    assert res["capacity"] == 0
    assert (res["row_of_slot"] == -1).all()
    assert res["dropped"].sum() == 4 and res["offsets"][-1] == 0


# --------------------------------------------------- top-k: brute force
def _unique_topk_set(keys, k):
    """The one k-subset where every chosen expert beats every other one:
    larger key, or equal key and lower index."""
    e = len(keys)
    found = []
    for sub in itertools.combinations(range(e), k):
        ok = all(keys[i] > keys[u] or (keys[i] == keys[u] and i < u)
                 for i in sub for u in range(e) if u not in sub)
        if ok:
            found.append(set(sub))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("n_exp,k", [(1, 1), (3, 1), (4, 2), (5, 3), (6, 2),
                                     (6, 3), (6, 6)])
@pytest.mark.parametrize("kind", ["ties", "normal", "signed_zero"])
def test_topk_brute_force(n_exp, k, kind):
    logits = W.make_logits(8, n_exp, seed=n_exp * 10 + k, kind=kind)
    idx = O.top_k(logits, k)
    for t in range(logits.shape[0]):
        keys = [float(v) for v in logits[t]]
        assert set(idx[t].tolist()) == _unique_topk_set(keys, k)
        for a, b in zip(idx[t][:-1], idx[t][1:]):
            assert keys[a] > keys[b] or (keys[a] == keys[b] and a < b)


def test_signed_zero_ties_go_to_lower_index():
    logits = np.array([[-0.0, 0.0, -0.0, -1.0]], np.float32)
    assert O.top_k(logits, 2).tolist() == [[0, 1]]
    logits = np.array([[0.0, -0.0, 0.0, -1.0]], np.float32)
    assert O.top_k(logits, 3).tolist() == [[0, 1, 2]]


def test_sigmoid_mode_brute_force_with_bias():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((8, 6)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, 6).astype(np.float32)
    idx, w, _ = O.route(logits, O.SIGMOID_BIAS, 3, bias)
    s = torch.sigmoid(torch.from_numpy(logits).double()).float().numpy()
    keys = (s + bias).astype(np.float32)
    for t in range(8):
        assert set(idx[t].tolist()) == _unique_topk_set(
            [float(v) for v in keys[t]], 3)
        ssel = s[t, idx[t]].astype(np.float64)
        # weights use the raw affinities, not the biased keys
        assert np.allclose(w[t], ssel / ssel.sum(), rtol=1e-12, atol=0)


def test_sigmoid_bias_changes_selection_but_not_weight_formula():
    logits = np.array([[2.0, 1.9, -3.0]], np.float32)
    bias = np.array([0.0, 0.0, 0.95], np.float32)
    idx, w, p = O.route(logits, O.SIGMOID_BIAS, 2, bias)
    assert idx.tolist() == [[2, 0]]          # bias promotes expert 2 to first
    s = 1.0 / (1.0 + np.exp(-np.array([-3.0, 2.0])))
    assert np.allclose(w[0], s / s.sum(), rtol=1e-6)
    assert np.allclose(p.sum(axis=1), 1.0)


# ------------------------------------------------------------- weights
@pytest.mark.parametrize("mode", [O.SOFTMAX_TOPK, O.TOPK_SOFTMAX])
def test_softmax_weights_sum_to_one_and_distinct(mode):
    """BUILD guide test: top-k weights sum to 1; DSEEK: k distinct experts."""
    logits = W.make_logits(64, 8, seed=5)
    idx, w, p = O.route(logits, mode, 2)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert all(len(set(r)) == 2 for r in idx.tolist())
    assert np.allclose(p.sum(axis=1), 1.0)


def test_two_softmax_modes_agree_and_match_torch():
    logits = W.make_logits(50, 16, seed=6)
    i1, w1, p1 = O.route(logits, O.SOFTMAX_TOPK, 4)
    i2, w2, p2 = O.route(logits, O.TOPK_SOFTMAX, 4)
    assert np.array_equal(i1, i2)
    assert np.allclose(w1, w2, rtol=1e-12, atol=1e-15)
    lt = torch.from_numpy(logits).double()
    assert np.allclose(p1, torch.softmax(lt, -1).numpy(), rtol=1e-12)
    tv, ti = torch.topk(lt, 4, dim=-1)
    assert np.array_equal(np.sort(i2, 1), np.sort(ti.numpy(), 1))
    ref = torch.softmax(tv, -1).numpy()
    assert np.allclose(w2, ref, rtol=1e-12)


def test_k_equals_e_weights_are_full_softmax():
    logits = W.make_logits(10, 5, seed=9)
    idx, w, _ = O.route(logits, O.SOFTMAX_TOPK, 5)
    full = torch.softmax(torch.from_numpy(logits).double(), -1).numpy()
    assert np.allclose(w, np.take_along_axis(full, idx, 1), rtol=1e-12)


# ------------------------------------------------------------- rounding
def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    a = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(
        -5, 5, 20000), [0.0, -0.0, 1.0, 3.0e38, -3.0e38]]).astype(np.float32)
    # exact bf16 halfway points (ties) in both directions
    hi = (rng.integers(100, 150, 1000).astype(np.uint32) << 7) | \
        rng.integers(0, 128, 1000).astype(np.uint32)
    u = (hi << 16) | np.uint32(0x8000)
    a = np.concatenate([a, u.view(np.float32), -u.view(np.float32)])
    ref = torch.from_numpy(a).to(torch.bfloat16).double().numpy()
    got = O.round_bf16(a.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_avoids_double_rounding():
    # 1 + 2^-8 + 2^-30 lies just above the bf16 midpoint between 1 and
    # 1 + 2^-7; fp32 rounding lands exactly on the midpoint, so a naive
    # double rounding would tie to even (1.0).  The correct answer is 1+2^-7.
    a = np.array([1 + 2.0 ** -8 + 2.0 ** -30, -(1 + 2.0 ** -8 + 2.0 ** -30),
                  1 + 2.0 ** -8 - 2.0 ** -30, 1 + 2.0 ** -8,
                  1 + 3 * 2.0 ** -8])
    got = O.round_bf16(a)
    assert got.tolist() == [1 + 2.0 ** -7, -(1 + 2.0 ** -7), 1.0, 1.0,
                            1 + 2 * 2.0 ** -7]


# --------------------------------------------------------------- pieces
def test_router_logits_of_unit_inputs_are_weight_columns():
    """BUILD step 2: the gate is Linear(d, E), logits = x W^T + b; a unit
    input picks one column of W (a transposed W would pick a row)."""
    w = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    b = np.array([0.5, -1.0])
    x = np.array([[0.0, 1.0, 0.0], [0.0, 0.0, 2.0]])
    assert O.router_logits(x, w, b).tolist() == [[2.5, 4.0], [6.5, 11.0]]
    assert O.router_logits(x, w).tolist() == [[2.0, 5.0], [6.0, 12.0]]


@pytest.mark.parametrize("mode", [O.SOFTMAX_TOPK, O.TOPK_SOFTMAX])
def test_softmax_mode_weights_closed_form(mode):
    """Logits ln(1, 2, 5, 1/2): top-2 is experts 2 and 1 with weights 5/7 and
    2/7 in both softmax modes (BUILD step 2; QWEN routing probabilities); the
    statistic's p is the full softmax, (1, 2, 5, 1/2) / 8.5."""
    lg = np.log(np.array([[1.0, 2.0, 5.0, 0.5]])).astype(np.float32)
    idx, w, p = O.route(lg, mode, 2)
    assert idx.tolist() == [[2, 1]]
    assert np.allclose(w, [[5 / 7, 2 / 7]], rtol=1e-6, atol=0)
    assert np.allclose(p, [[1 / 8.5, 2 / 8.5, 5 / 8.5, 0.5 / 8.5]], rtol=1e-6, atol=0)


def test_sigmoid_mode_weights_closed_form():
    """DSEEK s.2: logits ln(1, 3, 1/3, 7) give s = (1/2, 3/4, 1/4, 7/8).
    Without a bias, top-2 is experts 3 and 1 with weights 7/13 and 6/13; a
    bias of 0.7 on expert 2 selects experts 2 and 3, whose weights use s
    alone: 2/9 and 7/9.  p = s / sum(s) either way."""
    lg = np.log(np.array([[1.0, 3.0, 1 / 3, 7.0]])).astype(np.float32)
    p_want = [[0.5 / 2.375, 0.75 / 2.375, 0.25 / 2.375, 0.875 / 2.375]]
    idx, w, p = O.route(lg, O.SIGMOID_BIAS, 2, np.zeros(4, np.float32))
    assert idx.tolist() == [[3, 1]]
    assert np.allclose(w, [[7 / 13, 6 / 13]], rtol=1e-6, atol=0)
    assert np.allclose(p, p_want, rtol=1e-6, atol=0)
    idx, w, p = O.route(lg, O.SIGMOID_BIAS, 2, np.array([0, 0, 0.7, 0], np.float32))
    assert idx.tolist() == [[2, 3]]
    assert np.allclose(w, [[2 / 9, 7 / 9]], rtol=1e-6, atol=0)
    assert np.allclose(p, p_want, rtol=1e-6, atol=0)


def test_router_logits_match_torch_linear():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 5))
    w = rng.standard_normal((3, 5))
    b = rng.standard_normal(3)
    ref = TF.linear(torch.from_numpy(x), torch.from_numpy(w),
                    torch.from_numpy(b)).float().numpy()
    assert np.array_equal(O.router_logits(x, w, b), ref)


def test_silu_matches_torch():
    z = np.linspace(-50, 50, 1001)
    assert np.allclose(O.silu(z), TF.silu(torch.from_numpy(z)).numpy(),
                       rtol=1e-14, atol=1e-300)


def _torch_round(t, dtype):
    return t.to(torch.bfloat16 if dtype == O.BF16 else torch.float32).double()


@pytest.mark.parametrize("dtype", [O.F32, O.BF16])
@pytest.mark.parametrize("kind", [O.SILU_MLP, O.SWIGLU])
def test_expert_ffn_matches_torch(kind, dtype):
    rng = np.random.default_rng(4)
    d, f, m = 12, 20, 9
    x = rng.standard_normal((m, d))
    w1 = rng.standard_normal((f, d)) / math.sqrt(d)
    w3 = rng.standard_normal((f, d)) / math.sqrt(d)
    w2 = rng.standard_normal((d, f)) / math.sqrt(f)
    b1, b2 = rng.standard_normal(f), rng.standard_normal(d)
    T = torch.from_numpy
    if kind == O.SWIGLU:
        h = TF.silu(TF.linear(T(x), T(w1))) * TF.linear(T(x), T(w3))
        h = _torch_round(h, dtype)
        y = TF.linear(h, T(w2))
        h_got, got = O.expert_ffn(x, w1, w2, kind, dtype, w3=w3)
    else:
        h = _torch_round(TF.silu(TF.linear(T(x), T(w1), T(b1))), dtype)
        y = TF.linear(h, T(w2), T(b2))
        h_got, got = O.expert_ffn(x, w1, w2, kind, dtype, b1=b1, b2=b2)
    # h is stored in the layer dtype, y in fp32
    assert np.array_equal(h_got, h.numpy())
    ref = y.float().double().numpy()
    close = np.isclose(got, ref, rtol=1e-12, atol=0)
    assert close.mean() > 0.98
    assert np.all(np.abs(got - ref) <= 2 * 2.0 ** -23 * np.abs(ref) + 1e-300)


# Closed forms of the expert FFN.  The weights are scaled permutation
# matrices, so every output is one or two values of silu(z) = z * sigma(z) at
# z in {1, 2, -1}, written out below as decimal literals from the logistic
# function's values (sigma(1) = e / (1 + e), sigma(2) = e^2 / (1 + e^2),
# sigma(-1) = 1 - sigma(1)).  A swapped gate and up matrix, a transposed
# operand, a bias in the wrong place, a missing activation, a wrong rounding
# point or a wrong expert index each changes at least one of them.
SILU_1 = 0.7310585786300049          # silu(1) = sigma(1)
SILU_2 = 1.7615941559557646          # silu(2) = 2 sigma(2)
SILU_M1 = -0.2689414213699951        # silu(-1) = -(1 - sigma(1))


def _swiglu_closed_form_weights():
    # W1 x = (x1, x2, x0); W3 x = 0.5 (x2, x0, x1); y = (1.25 h2, 2 h0, 3 h1)
    w1 = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0]], np.float64)
    w3 = 0.5 * np.array([[0, 0, 1], [1, 0, 0], [0, 1, 0]], np.float64)
    w2 = np.array([[0, 0, 1.25], [2, 0, 0], [0, 3, 0]], np.float64)
    return w1, w3, w2


def test_swiglu_expert_closed_form_fp32():
    """QWEN expert forward pass / DSEEK s.1: h = silu(W1 x) * (W3 x), y = W2 h."""
    w1, w3, w2 = _swiglu_closed_form_weights()
    x = np.array([[1.0, 2.0, -1.0]])
    # W1 x = (2, -1, 1), W3 x = (-0.5, 0.5, 1)
    want_h = [-0.5 * SILU_2, 0.5 * SILU_M1, SILU_1]
    want_y = [1.25 * SILU_1, -SILU_2, 1.5 * SILU_M1]
    h, y = O.expert_ffn(x, w1, w2, O.SWIGLU, O.F32, w3=w3)
    assert np.allclose(h[0], want_h, rtol=1.2e-7, atol=0)
    assert np.allclose(y[0], want_y, rtol=2.5e-7, atol=0)


def test_swiglu_expert_closed_form_bf16_rounds_h_only():
    """bf16 layers store h in bf16 and accumulate y in fp32: h = bf16 of
    (-0.88080, -0.13447, 0.73106) = (-225/256, -138/1024, 187/256); y = W2 h
    is then exact in fp32 (1.25 * 187/256 = 233.75/256 is not a bf16 value,
    so rounding y to bf16 as well would show)."""
    w1, w3, w2 = _swiglu_closed_form_weights()
    x = np.array([[1.0, 2.0, -1.0]])
    h, y = O.expert_ffn(x, w1, w2, O.SWIGLU, O.BF16, w3=w3)
    assert h[0].tolist() == [-0.87890625, -0.134765625, 0.73046875]
    assert y[0].tolist() == [0.9130859375, -1.7578125, -0.404296875]


def test_silu_mlp_expert_closed_form_with_biases():
    """EXPERT In[7]: h = silu(W1 x + b1), y = W2 h + b2."""
    x = np.array([[0.5, -1.0]])
    w1 = np.array([[2.0, 0.0], [0.0, -1.0], [1.0, 1.0]])     # W1 x = (1, 1, -0.5)
    b1 = np.array([0.0, 1.0, 0.5])                           # pre-activation (1, 2, 0)
    w2 = np.array([[1.0, -1.0, 4.0], [0.0, 0.5, 0.0]])
    b2 = np.array([0.25, -1.0])
    h, y = O.expert_ffn(x, w1, w2, O.SILU_MLP, O.F32, b1=b1, b2=b2)
    assert np.allclose(h[0], [SILU_1, SILU_2, 0.0], rtol=1.2e-7, atol=0)
    assert np.allclose(y[0], [SILU_1 - SILU_2 + 0.25, 0.5 * SILU_2 - 1.0], rtol=2.5e-7, atol=0)
    # bf16: h = (187/256, 225/128, 0), y exact in fp32
    h, y = O.expert_ffn(x, w1, w2, O.SILU_MLP, O.BF16, b1=b1, b2=b2)
    assert h[0].tolist() == [0.73046875, 1.7578125, 0.0]
    assert y[0].tolist() == [-0.77734375, -0.12109375]


def test_grouped_ffn_applies_each_expert_to_its_own_rows():
    """d = F = 1: expert 0 is (w1, w3, w2) = (1, 1, 1), expert 1 is empty,
    expert 2 is (2, -1, 0.5); rows 0 | - | 1, 2 by the offsets."""
    p = {"w1": np.array([1.0, 9.0, 2.0]).reshape(3, 1, 1),
         "w3": np.array([1.0, 9.0, -1.0]).reshape(3, 1, 1),
         "w2": np.array([1.0, 9.0, 0.5]).reshape(3, 1, 1)}
    x = np.array([[1.0], [1.0], [-0.5]])
    _, y = O.grouped_ffn(x, [0, 1, 1, 3], p, O.SWIGLU, O.F32)
    # row 0: silu(1); row 1: 0.5 * silu(2) * (-1); row 2: 0.5 * silu(-1) * 0.5
    assert np.allclose(y[:, 0], [SILU_1, -0.5 * SILU_2, 0.25 * SILU_M1], rtol=2.5e-7, atol=0)


def test_combine_matches_index_add():
    rng = np.random.default_rng(8)
    n, k, d, e = 6, 3, 4, 5
    idx = np.stack([rng.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    disp = O.dispatch(idx, e, 0.0)
    m = int(disp["offsets"][-1])
    y = rng.standard_normal((m, d))
    w = rng.random((n, k))
    got = O.combine(y, disp["row_of_slot"], w)
    out = torch.zeros(n, d, dtype=torch.float64)
    rows = disp["row_of_slot"].reshape(n, k)
    for j in range(k):
        out.index_add_(0, torch.arange(n), torch.from_numpy(
            y[rows[:, j]] * w[:, j:j + 1]))
    assert np.allclose(got, out.numpy(), rtol=1e-14)


def test_combine_dropped_slot_contributes_zero():
    y = np.array([[1.0, 2.0]])
    got = O.combine(y, np.array([0, -1]), np.array([[0.25, 0.75]]))
    assert got.tolist() == [[0.25, 0.5]]


def test_shared_experts_concatenation_identity():
    rng = np.random.default_rng(10)
    d, fs, n = 8, 6, 5
    ws1 = rng.standard_normal((2, fs, d))
    ws3 = rng.standard_normal((2, fs, d))
    ws2 = rng.standard_normal((2, d, fs))
    x = rng.standard_normal((n, d))
    two = O.shared_ffn(x, ws1, ws3, ws2, O.F32)
    one = O.shared_ffn(x, ws1.reshape(1, 2 * fs, d), ws3.reshape(1, 2 * fs, d),
                       np.concatenate([ws2[0], ws2[1]], axis=1)[None], O.F32)
    assert np.allclose(two, one, rtol=1e-12, atol=1e-12)
    T = torch.from_numpy
    ref = sum(TF.linear(_torch_round(TF.silu(TF.linear(T(x), T(ws1[s]))) *
                                     TF.linear(T(x), T(ws3[s])), O.F32),
                        T(ws2[s])) for s in range(2))
    assert np.allclose(two, ref.numpy(), rtol=1e-6, atol=1e-9)


def test_shared_experts_closed_form():
    """DSEEK s.4: the shared experts are always on, each with weight 1, and
    their outputs add.  d = F_s = 1: expert 0 is (1, 1, 1), expert 1 is
    (2, -1, 0.5); x = 1 gives silu(1) + 0.5 * silu(2) * (-1)."""
    ws1 = np.array([1.0, 2.0]).reshape(2, 1, 1)
    ws3 = np.array([1.0, -1.0]).reshape(2, 1, 1)
    ws2 = np.array([1.0, 0.5]).reshape(2, 1, 1)
    x = np.array([[1.0]])
    got = O.shared_ffn(x, ws1, ws3, ws2, O.F32)
    assert np.allclose(got[0], [SILU_1 - 0.5 * SILU_2], rtol=1e-6, atol=0)
    # bf16: each expert's h is rounded (187/256 and -225/128), the sum is not
    assert O.shared_ffn(x, ws1, ws3, ws2, O.BF16)[0].tolist() == [0.73046875 - 0.87890625]


# ------------------------------------------------------ balance statistic
def test_balance_uniform_routing_closed_form():
    n, e, k, coef = 64, 8, 2, 0.01
    counts = np.full(e, n * k // e)
    p = np.full((n, e), 1.0 / e)
    assert math.isclose(O.balance_statistic(counts, p, n, coef),
                        coef * k / e, rel_tol=1e-12)


def test_balance_collapsed_routing_closed_form():
    # every token picks experts {0, 1} with p = 1/2 each: B = coef * 2*(1*1/2)
    n, e, coef = 16, 8, 0.01
    counts = np.zeros(e)
    counts[:2] = n
    p = np.zeros((n, e))
    p[:, :2] = 0.5
    assert math.isclose(O.balance_statistic(counts, p, n, coef), coef,
                        rel_tol=1e-12)


def test_balance_bounds_on_random_routing():
    logits = W.make_logits(100, 8, seed=12)
    idx, w, p = O.route(logits, O.SOFTMAX_TOPK, 2)
    res = O.dispatch(idx, 8, 0.0)
    b = O.balance_statistic(res["counts"], p, 100, 0.01)
    assert 0.0 <= b <= 0.01 * 2


# --------------------------------------------------- special-case layers
def _tiny_shape(**kw):
    base = dict(name="tiny", n_tokens=10, d_model=8, n_experts=4, top_k=2,
                d_ff=12, expert=W.EXPERT_SWIGLU, route=W.ROUTE_SOFTMAX_TOPK,
                dtype=W.DTYPE_F32, seed=21)
    base.update(kw)
    return W.MoEShape(**base)


def _torch_expert(x, v, e, kind, dtype):
    T = torch.from_numpy
    xx = T(x).double()
    if kind == W.EXPERT_SWIGLU:
        h = TF.silu(TF.linear(xx, T(v["w1"][e]).double())) * TF.linear(
            xx, T(v["w3"][e]).double())
        return TF.linear(_torch_round(h, dtype), T(v["w2"][e]).double()).float().double()
    h = TF.silu(TF.linear(xx, T(v["w1"][e]).double(), T(v["b1"][e]).double()))
    return TF.linear(_torch_round(h, dtype), T(v["w2"][e]).double(),
                     T(v["b2"][e]).double()).float().double()


@pytest.mark.parametrize("kind", [W.EXPERT_SWIGLU, W.EXPERT_SILU_MLP])
def test_single_expert_top1_is_dense_ffn(kind):
    shape = _tiny_shape(n_experts=1, top_k=1, expert=kind,
                        has_bias=kind == W.EXPERT_SILU_MLP)
    v = W.make_inputs(shape).values
    res = O.forward(shape, v)
    ref = _torch_expert(v["x"], v, 0, kind, W.DTYPE_F32).numpy()
    assert np.allclose(res["out"], ref, rtol=1e-6, atol=1e-7)
    assert (res["idx"] == 0).all() and np.allclose(res["w"], 1.0)


def test_k_equals_e_is_dense_all_expert_sum_with_shared():
    """DSEEK worked example: d=16, 4 experts, 1 shared; with k = E the sparse
    layer equals the dense all-expert weighted sum plus the shared expert."""
    shape = _tiny_shape(n_tokens=8, d_model=16, n_experts=4, top_k=4,
                        n_shared=1, d_ff_shared=12)
    v = W.make_inputs(shape).values
    res = O.forward(shape, v)
    assert res["out"].shape == (8, 16)
    T = torch.from_numpy
    logits = TF.linear(T(v["x"]).double(), T(v["w_router"]).double()).float()
    probs = torch.softmax(logits.double(), -1)
    dense = sum(probs[:, e:e + 1] * _torch_expert(v["x"], v, e, W.EXPERT_SWIGLU,
                                                   W.DTYPE_F32)
                for e in range(4))
    xx = T(v["x"]).double()
    sh = TF.linear(_torch_round(TF.silu(TF.linear(xx, T(v["ws1"][0]).double()))
                                * TF.linear(xx, T(v["ws3"][0]).double()),
                                W.DTYPE_F32), T(v["ws2"][0]).double())
    ref = (dense + sh.float().double()).float().numpy()
    assert np.allclose(res["out"], ref, rtol=1e-5, atol=1e-6)


def test_top2_worked_example_invariants():
    """DSEEK worked example: B=2, T=4, d=16, 4 experts, top-2, 1 shared."""
    shape = _tiny_shape(n_tokens=8, d_model=16, n_experts=4, top_k=2,
                        n_shared=1, d_ff_shared=12)
    v = W.make_inputs(shape).values
    res = O.forward(shape, v)
    assert res["out"].shape == (8, 16)
    assert res["idx"].shape == (8, 2)
    assert all(len(set(r)) == 2 for r in res["idx"].tolist())
    assert res["counts"].sum() == 16
    assert np.array_equal(np.sort(res["row_of_slot"]), np.arange(16))


def test_forward_tokens_matches_forward():
    shape = _tiny_shape(n_tokens=12, n_experts=5, top_k=3, dtype=W.DTYPE_BF16,
                        route=W.ROUTE_SIGMOID_BIAS, sel_bias_range=0.1,
                        n_shared=2, d_ff_shared=8)
    v = W.make_inputs(shape).values
    full = O.forward(shape, v)
    part = O.forward_tokens(shape, v, [0, 5, 11])
    assert np.array_equal(part["idx"], full["idx"][[0, 5, 11]])
    assert np.allclose(part["out"], full["out"][[0, 5, 11]], rtol=0, atol=1e-2)


# ---------------------------------------------- selection-bias update, CV
def test_bias_update_moves_against_the_load():
    """Over-loaded experts lose gamma, under-loaded gain it, one at the mean
    keeps its bias (mean of (6, 2, 4, 4) is 4)."""
    b = np.array([0.5, -0.25, 0.0, 0.125], np.float32)
    got = O.selection_bias_update(b, [6, 2, 4, 4], 0.01)
    g = np.float32(0.01)
    assert got.dtype == np.float32
    assert got[0] == np.float32(0.5) - g and got[1] == np.float32(-0.25) + g
    assert got[2] == np.float32(0.0) and got[3] == np.float32(0.125)


def test_bias_update_fixed_points():
    b = np.random.default_rng(0).uniform(-0.1, 0.1, 16).astype(np.float32)
    assert np.array_equal(O.selection_bias_update(b, np.full(16, 7), 0.5), b)   # balanced
    assert np.array_equal(O.selection_bias_update(b, np.zeros(16, int), 0.5), b)  # nothing routed
    assert np.array_equal(O.selection_bias_update(b, [3] * 16, 0.0), b)


def test_bias_update_sign_decided_exactly():
    # mean load 10/3 is not a float; the sign compares E * load with the
    # total on integers: 9 < 10 (below), 12 > 10 (above)
    got = O.selection_bias_update(np.zeros(3, np.float32), [3, 3, 4], 1.0)
    assert list(got) == [1.0, 1.0, -1.0]


def test_load_cv_closed_forms():
    assert O.load_cv([5, 5, 5, 5]) == 0.0
    assert O.load_cv([0, 0, 0]) == 0.0
    # (1, 2, 3, 4): mean 2.5, population variance 1.25
    assert abs(O.load_cv([1, 2, 3, 4]) - np.sqrt(1.25) / 2.5) < 1e-15
    # everything on one of E experts: cv = sqrt(E - 1)
    assert abs(O.load_cv([0, 0, 0, 0, 0, 0, 0, 80]) - np.sqrt(7.0)) < 1e-12
