"""Pins of the backward oracle (CPU only).

The oracle's gradients are checked against central finite differences of a
fixed-route loss written here independently of it (plain loops over tokens
and slots), and against properties the pages and the mathematics fix: an
expert no token selected gets no gradient, a dropped assignment passes no
gradient to its expert, the softmax-mode logit gradients sum to zero per
token, and the two softmax modes are the same function.
"""
import numpy as np
import pytest

from oracle import moe_backward as B
from oracle import moe_oracle as O
from routing_dispatch_expert_05_b300 import workloads as W


def _shape(route=W.ROUTE_SOFTMAX_TOPK, expert=W.EXPERT_SWIGLU, n_shared=0, cf=0.0,
           bias=False, router_bias="normal", N=7, d=8, E=5, k=2, F=4, seed=11):
    return W.MoEShape(name="bwd", n_tokens=N, d_model=d, n_experts=E, top_k=k, d_ff=F,
                      expert=expert, route=route, dtype=W.DTYPE_F32, has_bias=bias,
                      router_bias=router_bias, sel_bias_range=0.2, capacity_factor=cf,
                      n_shared=n_shared, d_ff_shared=4 if n_shared else 0,
                      balance_coef=0.3, seed=seed)


def _values64(shape):
    v = W.make_inputs(shape).values
    return {key: np.asarray(a, np.float64) for key, a in v.items()}


def _loss(shape, v, dout, d_balance, idx, kept, counts):
    """<dout, out> + d_balance * B for fixed routing, one token and slot at a
    time."""
    x = v["x"]
    n, d = x.shape
    z = x @ v["w_router"].T
    if "b_router" in v:
        z = z + v["b_router"]
    total = 0.0
    p_sum = np.zeros(shape.n_experts)
    for t in range(n):
        zt = z[t]
        if shape.route == W.ROUTE_SIGMOID_BIAS:
            s = 1.0 / (1.0 + np.exp(-zt))
            sel = s[idx[t]]
            wt = sel / sel.sum()
            p_sum += s / s.sum()
        else:
            ez = np.exp(zt - zt.max())
            p_full = ez / ez.sum()
            if shape.route == W.ROUTE_SOFTMAX_TOPK:
                sel = p_full[idx[t]]
                wt = sel / sel.sum()
            else:
                es = np.exp(zt[idx[t]] - zt[idx[t]].max())
                wt = es / es.sum()
            p_sum += p_full
        out = np.zeros(d)
        for j in range(shape.top_k):
            if not kept[t, j]:
                continue
            e = idx[t, j]
            g = v["w1"][e] @ x[t]
            if shape.expert == W.EXPERT_SWIGLU:
                h = g / (1.0 + np.exp(-g)) * (v["w3"][e] @ x[t])
            else:
                if "b1" in v:
                    g = g + v["b1"][e]
                h = g / (1.0 + np.exp(-g))
            y = v["w2"][e] @ h
            if "b2" in v:
                y = y + v["b2"][e]
            out += wt[j] * y
        for s_ in range(shape.n_shared):
            g = v["ws1"][s_] @ x[t]
            out += v["ws2"][s_] @ (g / (1.0 + np.exp(-g)) * (v["ws3"][s_] @ x[t]))
        total += dout[t] @ out
    bal = shape.balance_coef * np.sum(np.asarray(counts) / n * p_sum / n)
    return total + d_balance * bal


CASES = [
    dict(route=W.ROUTE_SOFTMAX_TOPK),
    dict(route=W.ROUTE_TOPK_SOFTMAX, n_shared=1),
    dict(route=W.ROUTE_SIGMOID_BIAS, n_shared=1),
    dict(route=W.ROUTE_SOFTMAX_TOPK, expert=W.EXPERT_SILU_MLP, bias=True),
    dict(route=W.ROUTE_SOFTMAX_TOPK, expert=W.EXPERT_SILU_MLP, bias=True, cf=1.0, N=10),
    dict(route=W.ROUTE_SIGMOID_BIAS, cf=1.0, N=10, k=3, router_bias="none"),
]


@pytest.mark.parametrize("d_balance", [0.0, 2.5])
@pytest.mark.parametrize("case", CASES)
def test_backward_matches_finite_differences(case, d_balance):
    shape = _shape(**case)
    v = _values64(shape)
    rng = np.random.default_rng(5)
    dout = rng.standard_normal((shape.n_tokens, shape.d_model))
    fixed = B.fixed_route(shape, v)
    idx, kept, counts = fixed
    if case.get("cf"):
        assert not kept.all()                    # the capacity drops something
    g = B.layer_backward(shape, v, dout, d_balance, route_fixed=fixed)
    names = {"x": "dx", "w_router": "d_w_router", "b_router": "d_b_router", "w1": "d_w1",
             "w3": "d_w3", "w2": "d_w2", "b1": "d_b1", "b2": "d_b2", "ws1": "d_ws1",
             "ws3": "d_ws3", "ws2": "d_ws2"}
    eps = 1e-6
    checked = 0
    for pname, gname in names.items():
        if pname not in v:
            continue
        a = v[pname]
        for flat in rng.choice(a.size, size=min(6, a.size), replace=False):
            pos = np.unravel_index(flat, a.shape)
            keep = a[pos]
            a[pos] = keep + eps
            lp = _loss(shape, v, dout, d_balance, idx, kept, counts)
            a[pos] = keep - eps
            lm = _loss(shape, v, dout, d_balance, idx, kept, counts)
            a[pos] = keep
            fd = (lp - lm) / (2 * eps)
            assert abs(g[gname][pos] - fd) <= 1e-6 * max(1.0, abs(fd)), (pname, pos)
            checked += 1
    assert checked >= 30


def test_unused_expert_gets_no_gradient():
    shape = _shape(N=9, E=6, k=2)
    v = _values64(shape)
    v["b_router"][4] = -50.0                      # nobody selects expert 4
    dout = np.random.default_rng(1).standard_normal((shape.n_tokens, shape.d_model))
    idx, kept, counts = B.fixed_route(shape, v)
    assert counts[4] == 0
    g = B.layer_backward(shape, v, dout, 1.0)
    for name in ("d_w1", "d_w3", "d_w2"):
        assert np.all(g[name][4] == 0.0), name
    assert np.any(g["d_w1"][idx[0, 0]] != 0.0)


def test_dropped_assignment_passes_no_gradient_to_its_expert():
    shape = _shape(N=12, E=3, k=2, cf=0.5)      # capacity 2 per expert
    v = _values64(shape)
    dout = np.random.default_rng(2).standard_normal((shape.n_tokens, shape.d_model))
    idx, kept, counts = B.fixed_route(shape, v)
    assert (~kept).sum() > 0
    g = B.layer_backward(shape, v, dout)
    assert np.all(g["dy"][~kept] == 0.0) and np.all(g["dw"][~kept] == 0.0)
    # the expert weight gradients are those of the kept rows alone: each
    # expert sees at most `capacity` rows
    cap = O.capacity(shape.capacity_factor, shape.n_tokens, shape.n_experts)
    assert int(kept.sum()) <= cap * shape.n_experts


@pytest.mark.parametrize("mode", [W.ROUTE_SOFTMAX_TOPK, W.ROUTE_TOPK_SOFTMAX])
def test_softmax_mode_logit_gradients_sum_to_zero(mode):
    shape = _shape(route=mode, N=8, E=6, k=3)
    v = _values64(shape)
    dout = np.random.default_rng(3).standard_normal((shape.n_tokens, shape.d_model))
    g = B.layer_backward(shape, v, dout, 4.0)
    assert np.abs(g["dlogits"].sum(axis=1)).max() < 1e-12
    assert np.abs(g["dlogits"]).max() > 1e-3


def test_both_softmax_modes_give_the_same_gradients():
    s0 = _shape(route=W.ROUTE_SOFTMAX_TOPK, N=8, E=6, k=3)
    s1 = s0.replace(route=W.ROUTE_TOPK_SOFTMAX)
    v = _values64(s0)
    dout = np.random.default_rng(4).standard_normal((s0.n_tokens, s0.d_model))
    g0 = B.layer_backward(s0, v, dout, 1.5)
    g1 = B.layer_backward(s1, v, dout, 1.5)
    for name in ("dx", "d_w_router", "d_w1", "d_w2", "d_w3", "dlogits"):
        assert np.allclose(g0[name], g1[name], rtol=1e-12, atol=1e-14), name


def test_dense_case_router_gradient_closed_form():
    """k = E: the routed output is the softmax mixture sum_e p_e y_e, whose
    logit gradient is p_e (<dout, y_e> - <dout, out_routed>)."""
    shape = _shape(route=W.ROUTE_TOPK_SOFTMAX, N=5, E=4, k=4)
    v = _values64(shape)
    dout = np.random.default_rng(6).standard_normal((shape.n_tokens, shape.d_model))
    g = B.layer_backward(shape, v, dout)
    x = v["x"]
    z = x @ v["w_router"].T + v["b_router"]
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    for t in range(shape.n_tokens):
        ys = []
        for e in range(shape.n_experts):
            gg = v["w1"][e] @ x[t]
            ys.append(v["w2"][e] @ (gg / (1 + np.exp(-gg)) * (v["w3"][e] @ x[t])))
        ys = np.array(ys)
        r = dout[t] @ ys.T                          # <dout, y_e>
        want = p[t] * (r - p[t] @ r)
        assert np.allclose(g["dlogits"][t], want, rtol=1e-10, atol=1e-12)
