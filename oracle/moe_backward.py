"""CPU oracle for the backward pass of the sparse-MoE FFN layer -- TEST
INFRASTRUCTURE ONLY.

Only the tests may use this module.  It shares no code with the CUDA
library; like the forward oracle it is plain float64 NumPy, written for
reading, not speed.

What it computes.  The pages fix the properties of the backward, not its
formulas ("DeepSeek 5.7: MoE from scratch", Worked example: the router
receives gradients and an expert that a token did not select receives none
of that token's gradient; its study-lab exercises: the top-k selection
itself is not differentiable).  The plainest reading, used here: the gradient of

    L = <dout, out> + d_balance * B

with the routing decisions held fixed -- which experts each token selected
(taken from the forward, on its fp32 logits) and which assignments the
capacity kept.  Everything else is differentiated exactly, in float64 and
without the forward's storage roundings:

* the contribution weights as functions of the logits: the softmax over
  the selected logits in both softmax modes (SOFTMAX_TOPK renormalised over
  the k equals TOPK_SOFTMAX), s_sel / sum(s_sel) with s = sigmoid(logit) in
  the sigmoid mode (the selection bias only selects);
* the balance statistic B = coef * sum_e frac_e * mean_t p[t, e] through p
  (frac_e, a count, is constant): p = softmax(logits), or s / sum(s) in the
  sigmoid mode;
* a dropped assignment contributes nothing, but its weight still takes part
  in normalising the token's other weights (the forward does not
  renormalise after drops);
* experts (SwiGLU: y = W2 (silu(W1 x) * (W3 x)); SiLU-MLP: y = W2 silu(W1 x
  + b1) + b2) and the shared experts (weight 1) by the chain rule.

Parity status: pinned in ``tests/test_backward_oracle.py`` by central finite
differences of an independently written fixed-route loss, exact zeros for
unused experts and dropped assignments, and closed-form identities (the
softmax-mode logit gradients sum to zero per token; both softmax modes give
the same gradients).
"""
from __future__ import annotations

import numpy as np

from oracle.moe_oracle import (SIGMOID_BIAS, SWIGLU, dispatch, route,
                               router_logits)


def _f64(a):
    return None if a is None else np.asarray(a, np.float64)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _silu_and_grad(z):
    s = _sigmoid(z)
    return z * s, s * (1.0 + z * (1.0 - s))


def fixed_route(shape, values: dict):
    """The routing decisions of the forward: idx [N, k] and the kept mask
    [N, k] (False = dropped by the capacity)."""
    logits = router_logits(values["x"], values["w_router"], values.get("b_router"))
    idx, _, _ = route(logits, shape.route, shape.top_k, values.get("sel_bias"))
    disp = dispatch(idx, shape.n_experts, shape.capacity_factor)
    kept = (disp["row_of_slot"] >= 0).reshape(idx.shape)
    return idx.astype(np.int64), kept, disp["counts"]


def _weights_and_p(z, idx, mode):
    """w [N, k] over the selected logits and p [N, E] for the statistic."""
    z_sel = np.take_along_axis(z, idx, axis=1)
    if mode == SIGMOID_BIAS:
        s = _sigmoid(z)
        s_sel = np.take_along_axis(s, idx, axis=1)
        return s_sel / s_sel.sum(axis=1, keepdims=True), s / s.sum(axis=1, keepdims=True)
    e_sel = np.exp(z_sel - z_sel.max(axis=1, keepdims=True))
    ez = np.exp(z - z.max(axis=1, keepdims=True))
    return e_sel / e_sel.sum(axis=1, keepdims=True), ez / ez.sum(axis=1, keepdims=True)


def layer_backward(shape, values: dict, dout, d_balance: float = 0.0, route_fixed=None):
    """Gradients of L = <dout, out> + d_balance * B (routing held fixed).

    Returns a dict with dx [N, d], d_w_router [E, d], d_b_router [E] (when
    the router has a bias), the expert weight gradients under the forward's
    names (d_w1, d_w3, d_w2, d_b1, d_b2), the shared ones (d_ws1, d_ws3,
    d_ws2), and the intermediates dlogits [N, E], dw [N, k] and dy [N, k, d]
    (the gradient reaching each assignment's expert output).
    """
    x = _f64(values["x"])
    n, d = x.shape
    n_exp, k, mode = shape.n_experts, shape.top_k, shape.route
    dout = _f64(dout)
    idx, kept, counts = route_fixed if route_fixed is not None else fixed_route(shape, values)

    wr = _f64(values["w_router"])
    br = _f64(values.get("b_router"))
    z = x @ wr.T + (br[None, :] if br is not None else 0.0)
    w, p = _weights_and_p(z, idx, mode)

    grads = {}
    dx = np.zeros_like(x)
    dw = np.zeros((n, k))
    dy = np.zeros((n, k, d))
    swiglu = shape.expert == SWIGLU
    w1, w2 = _f64(values["w1"]), _f64(values["w2"])
    w3 = _f64(values.get("w3"))
    b1, b2 = _f64(values.get("b1")), _f64(values.get("b2"))
    g_w1, g_w2 = np.zeros_like(w1), np.zeros_like(w2)
    g_w3 = np.zeros_like(w3) if w3 is not None else None
    g_b1 = np.zeros_like(b1) if b1 is not None else None
    g_b2 = np.zeros_like(b2) if b2 is not None else None

    # each kept assignment (t, j) -> expert e = idx[t, j]
    for t in range(n):
        a = x[t]
        for j in range(k):
            if not kept[t, j]:
                continue
            e = int(idx[t, j])
            g = w1[e] @ a
            if swiglu:
                u = w3[e] @ a
                sg, dsg = _silu_and_grad(g)
                h = sg * u
            else:
                if b1 is not None:
                    g = g + b1[e]
                sg, dsg = _silu_and_grad(g)
                h = sg
            y = w2[e] @ h
            if b2 is not None:
                y = y + b2[e]
            dw[t, j] = dout[t] @ y                  # out_t = sum_j w_tj y_tj
            dyj = w[t, j] * dout[t]
            dy[t, j] = dyj
            dh = w2[e].T @ dyj                      # y = W2 h (+ b2)
            g_w2[e] += np.outer(dyj, h)
            if g_b2 is not None:
                g_b2[e] += dyj
            if swiglu:
                dg = dh * u * dsg
                du = dh * sg
                g_w3[e] += np.outer(du, a)
                dx[t] += w3[e].T @ du
            else:
                dg = dh * dsg
                if g_b1 is not None:
                    g_b1[e] += dg
            g_w1[e] += np.outer(dg, a)
            dx[t] += w1[e].T @ dg

    # router: the weights' dependence on the selected logits
    dz = np.zeros((n, n_exp))
    wdw = np.sum(w * dw, axis=1, keepdims=True)
    if mode == SIGMOID_BIAS:
        s = _sigmoid(z)
        s_sel = np.take_along_axis(s, idx, axis=1)
        ds_sel = (dw - wdw) / s_sel.sum(axis=1, keepdims=True)
        np.put_along_axis(dz, idx, ds_sel * s_sel * (1.0 - s_sel), axis=1)
    else:
        np.put_along_axis(dz, idx, w * (dw - wdw), axis=1)
    # and the balance statistic's, through p
    if d_balance != 0.0 and n > 0:
        frac = np.asarray(counts, np.float64) / n
        gp = d_balance * shape.balance_coef * frac / n        # dB/dp[t, e]
        pg = np.sum(p * gp[None, :], axis=1, keepdims=True)
        if mode == SIGMOID_BIAS:
            s = _sigmoid(z)
            ds = (gp[None, :] - pg) / s.sum(axis=1, keepdims=True)
            dz += ds * s * (1.0 - s)
        else:
            dz += p * (gp[None, :] - pg)
    dx += dz @ wr
    grads["d_w_router"] = dz.T @ x
    if br is not None:
        grads["d_b_router"] = dz.sum(axis=0)

    if shape.n_shared > 0:
        ws1, ws3, ws2 = _f64(values["ws1"]), _f64(values["ws3"]), _f64(values["ws2"])
        g_ws1, g_ws3, g_ws2 = np.zeros_like(ws1), np.zeros_like(ws3), np.zeros_like(ws2)
        for s_ in range(ws1.shape[0]):
            g = x @ ws1[s_].T
            u = x @ ws3[s_].T
            sg, dsg = _silu_and_grad(g)
            h = sg * u
            dh = dout @ ws2[s_]
            g_ws2[s_] = dout.T @ h
            dg = dh * u * dsg
            du = dh * sg
            g_ws1[s_] = dg.T @ x
            g_ws3[s_] = du.T @ x
            dx += dg @ ws1[s_] + du @ ws3[s_]
        grads.update(d_ws1=g_ws1, d_ws3=g_ws3, d_ws2=g_ws2)

    grads.update(dx=dx, d_w1=g_w1, d_w2=g_w2, dlogits=dz, dw=dw, dy=dy)
    if g_w3 is not None:
        grads["d_w3"] = g_w3
    if g_b1 is not None:
        grads["d_b1"] = g_b1
    if g_b2 is not None:
        grads["d_b2"] = g_b2
    return grads
