"""CPU oracle for the sparse-MoE FFN forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module.  It shares no code with the CUDA library and imports nothing
from it; it is a plain, slow, obviously-correct statement of what the layer
computes, in float64 with the storage roundings the layer fixes.

Page citations (titles as printed on the pages):

* [BUILD]  "Hands-on build guide: pure-Python MoE router with load-balanced
  top-k gating": Architecture Overview; steps 2 (gate), 5 (combine);
  "Running and Testing It" step 3 (weights sum to 1).
* [EXPERT] "Expert Networks > Code Implementation": In[7] (SiLU-MLP expert
  with biases), In[8]/Out[9] (parameter count), In[10] (capacity and token
  dropping), Out[12] (capacity table), Out[15] (drop rate vs capacity).
* [DSEEK]  "DeepSeek 5.7: MoE from scratch": sections 1-4 (SwiGLU expert,
  sigmoid selection with a selection-only bias, dispatch/combine, shared
  experts), Worked example, Failure modes.
* [SER]    "Tutorial -- MoE SER Expert Routing": sections 3-4 (tokens per
  expert, load-balancing statistic coef * sum(frac * p_avg)).
* [QWEN]   "Implementing Mixed Expert (MoE) layers": Core Algorithmic Steps
  (topk on raw scores, softmax over the k, group by expert, SwiGLU expert,
  index_add_ combine).

Readings where the pages are silent or disagree (each also listed in the
design notes): storage points are x, weights, h and the output in the layer
dtype, logits, weights w, the expert outputs y and the shared sum S in
fp32; capacity is int(cf * (N // E)) applied per expert with
assignments taken in token order; dropped assignments contribute zero and the
surviving weights are not renormalised; ties go to the lowest expert index;
the softmax modes select on the raw logit; the sigmoid is evaluated in
float64 and rounded to fp32 before the fp32 bias add; frac_e counts
selections before any drop; the balance statistic's p is the full softmax
(softmax modes) or s / sum(s) (sigmoid mode); shared experts have weight 1.

Parity status: routing, dispatch, capacity, parameter count, balance
statistic and the FFN/combine structure are pinned by the tests under
``tests/test_oracle_pins.py``; the pages print no output values for the
FFN itself, so those values are pinned only through library routines and
special cases (dense FFN at E=1, all-expert sum at k=E), not by printed
numbers.
"""
from __future__ import annotations

import numpy as np

SOFTMAX_TOPK = 0
TOPK_SOFTMAX = 1
SIGMOID_BIAS = 2
SILU_MLP = 0
SWIGLU = 1
F32 = 0
BF16 = 1


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------
def round_bf16(a) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), as float64.

    Goes through fp32 first only when that is exact for the decision: a
    value is rounded to fp32 with round-to-nearest, then its low 16 bits are
    rounded away with round-to-nearest-even.  Double rounding can differ
    from a direct float64->bf16 rounding only when the fp32 rounding lands
    exactly on a bf16 tie; to avoid that, the tie case is decided on the
    float64 value.
    """
    a = np.asarray(a, dtype=np.float64)
    f = a.astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    low = u & 0xFFFF
    hi = u >> 16
    up = low > 0x8000
    tie = low == 0x8000
    # on an fp32-level tie, look at where the float64 value really lies
    f_back = f.astype(np.float64)
    above = a > f_back          # true value beyond the fp32 point, away from 0?
    below = a < f_back
    pos = (u >> 31) == 0
    # magnitude direction: for positive numbers "above" means larger magnitude
    larger_mag = np.where(pos, above, below)
    smaller_mag = np.where(pos, below, above)
    tie_up = tie & (larger_mag | (~smaller_mag & ((hi & 1) == 1)))
    hi = hi + (up | tie_up).astype(np.uint64)
    out = (hi << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    # keep non-finite values as they are
    bad = ~np.isfinite(a)
    if bad.any():
        out[bad] = a[bad]
    return out


def round_f32(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(dtype: int, a) -> np.ndarray:
    return round_bf16(a) if dtype == BF16 else round_f32(a)


# --------------------------------------------------------------------------
# the pieces of the layer
# --------------------------------------------------------------------------
def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))  [EXPERT In[7]; QWEN]."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_param_count(d_model: int, d_ff: int, bias: bool,
                       swiglu: bool = False) -> int:
    """Parameters of one expert: the shapes of its weight and bias tensors.

    SiLU-MLP: w1 [F, d] (+ b1 [F]), w2 [d, F] (+ b2 [d])   [EXPERT In[7]].
    SwiGLU adds the up projection w3 [F, d]                  [QWEN].
    """
    shapes = [(d_ff, d_model), (d_model, d_ff)]
    if swiglu:
        shapes.append((d_ff, d_model))
    if bias:
        shapes += [(d_ff,), (d_model,)]
    return int(sum(np.prod(s) for s in shapes))


def router_logits(x, w_router, b_router=None) -> np.ndarray:
    """logits[t, e] = sum_i x[t, i] * W[e, i] + b[e]; float64, stored fp32.

    The gate is one Linear(d, E) layer [BUILD step 2; QWEN gate computation].
    """
    z = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if b_router is not None:
        z = z + np.asarray(b_router, np.float64)[None, :]
    return z.astype(np.float32)


def softmax_rows(z) -> np.ndarray:
    z = np.asarray(z, np.float64)
    m = z.max(axis=1, keepdims=True)
    ez = np.exp(z - m)
    return ez / ez.sum(axis=1, keepdims=True)


def sigmoid_f32(logits) -> np.ndarray:
    """s = sigmoid(l) evaluated in float64 and rounded to fp32 [DSEEK s.2]."""
    l = np.asarray(logits, np.float32).astype(np.float64)
    with np.errstate(over="ignore"):
        return (1.0 / (1.0 + np.exp(-l))).astype(np.float32)


def selection_keys(logits, mode: int, sel_bias=None) -> np.ndarray:
    """The fp32 value experts are ranked by.

    Softmax modes rank by the raw logit (softmax is monotone, so the selected
    set is the one softmax would pick) [BUILD step 2; QWEN top-k].  The
    sigmoid mode ranks by sigmoid(l) + b with b used for selection only
    [DSEEK s.2]; the add is an fp32 add.
    """
    l = np.asarray(logits, np.float32)
    if mode == SIGMOID_BIAS:
        return (sigmoid_f32(l) + np.asarray(sel_bias, np.float32)[None, :]
                ).astype(np.float32)
    return l.copy()


def top_k(keys, k: int) -> np.ndarray:
    """Per row, the k experts of largest key; ties go to the lower index.

    Slot j holds the j-th best: key descending, index ascending.  A stable
    sort of the negated keys gives exactly that order (negation is exact and
    -0 == +0 compare equal, so they tie).
    """
    keys = np.asarray(keys, np.float32)
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def route(logits, mode: int, k: int, sel_bias=None):
    """Selection and contribution weights for each token.

    Returns ``idx [N,k]`` (int32), ``w [N,k]`` (float64) and ``p [N,E]``
    (float64), the per-token probabilities the balance statistic averages.

    * SOFTMAX_TOPK: p = softmax over all E; pick top-k; w = p_sel / sum p_sel
      [BUILD step 2 and its weights-sum-to-1 test].
    * TOPK_SOFTMAX: pick top-k logits; w = softmax over the k selected logits
      [QWEN top-k and routing probabilities]; p = softmax over all E.
    * SIGMOID_BIAS: s = sigmoid(l); pick top-k of s + b; w = s_sel / sum s_sel
      (bias excluded from the weight) [DSEEK s.2]; p = s / sum(s).
    """
    l = np.asarray(logits, np.float32)
    keys = selection_keys(l, mode, sel_bias)
    idx = top_k(keys, k)
    if mode == SIGMOID_BIAS:
        s = sigmoid_f32(l).astype(np.float64)
        s_sel = np.take_along_axis(s, idx, axis=1)
        w = s_sel / s_sel.sum(axis=1, keepdims=True)
        p = s / s.sum(axis=1, keepdims=True)
    else:
        p = softmax_rows(l)
        if mode == SOFTMAX_TOPK:
            p_sel = np.take_along_axis(p, idx, axis=1)
            w = p_sel / p_sel.sum(axis=1, keepdims=True)
        else:
            w = softmax_rows(np.take_along_axis(l.astype(np.float64), idx, axis=1))
    return idx, w, p


def capacity(capacity_factor: float, n_tokens: int, n_experts: int):
    """capacity = int(capacity_factor * (N // E)) [EXPERT In[10]]; None = no limit."""
    if capacity_factor is None or capacity_factor <= 0:
        return None
    return int(capacity_factor * (n_tokens // n_experts))


def dispatch(idx, n_experts: int, capacity_factor: float = 0.0, expert_capacity=None):
    """Group assignments by expert with a per-expert capacity [EXPERT In[10]].

    Assignments are visited in token order (and slot order within a token).
    An assignment to expert e is kept while e has processed fewer than
    ``capacity`` assignments, otherwise it is dropped and counted.  Kept
    assignments of expert e occupy rows offsets[e] .. offsets[e+1]-1 of the
    expert-sorted buffer in arrival order (a stable grouping) [DSEEK s.3;
    QWEN group tokens by expert].

    ``expert_capacity`` ([E] integers), if given, replaces the one capacity
    derived from ``capacity_factor`` by one per expert: what a shard of a
    larger batch may still keep once the assignments of the tokens before it
    are counted (the same token-order rule applied to the whole batch).

    Returns a dict with counts (selections per expert), kept, dropped,
    offsets [E+1], row_of_slot [N*k] (-1 = dropped) and token_of_row [M].
    """
    idx = np.asarray(idx, np.int64)
    n_tokens, k = idx.shape
    if expert_capacity is not None:
        caps = np.asarray(expert_capacity, np.int64)
        cap = None
    else:
        cap = capacity(capacity_factor, n_tokens, n_experts)
        caps = None
    counts = np.zeros(n_experts, np.int64)
    processed = np.zeros(n_experts, np.int64)
    dropped = np.zeros(n_experts, np.int64)
    local = np.full(n_tokens * k, -1, np.int64)
    flat = idx.reshape(-1).tolist()
    for s, e in enumerate(flat):
        counts[e] += 1
        limit = caps[e] if caps is not None else cap
        if limit is None or processed[e] < limit:
            local[s] = processed[e]
            processed[e] += 1
        else:
            dropped[e] += 1
    offsets = np.zeros(n_experts + 1, np.int64)
    offsets[1:] = np.cumsum(processed)
    row_of_slot = np.where(local >= 0, offsets[idx.reshape(-1)] + local, -1)
    m = int(offsets[-1])
    token_of_row = np.full(m, -1, np.int64)
    kept_slots = np.nonzero(row_of_slot >= 0)[0]
    token_of_row[row_of_slot[kept_slots]] = kept_slots // k
    return dict(capacity=caps if caps is not None else cap, counts=counts, kept=processed,
                dropped=dropped,
                offsets=offsets, row_of_slot=row_of_slot,
                token_of_row=token_of_row)


def permute_rows(x, token_of_row) -> np.ndarray:
    """x_perm[row] = x[token_of_row[row]] (gather by expert) [QWEN]."""
    return np.asarray(x)[np.asarray(token_of_row, np.int64)]


def expert_ffn(x_rows, w1, w2, kind: int, dtype: int, w3=None, b1=None,
               b2=None):
    """One expert applied to a block of rows; returns (h, y).

    SiLU-MLP: h = silu(W1 x + b1), y = W2 h + b2   [EXPERT In[7]].
    SwiGLU:   h = silu(W1 x) * (W3 x), y = W2 h     [QWEN expert forward pass;
              DSEEK s.1].
    h is rounded to the layer's storage type (bf16 or fp32).  y is rounded
    to fp32 only: it is an fp32 accumulation that feeds the weighted
    combine, itself part of the same fp32 accumulation (the layer is "bf16
    weights/activations, fp32 accumulation"), and the layer output is
    rounded once, at the end.
    """
    x = np.asarray(x_rows, np.float64)
    a = x @ np.asarray(w1, np.float64).T
    if kind == SWIGLU:
        h = silu(a) * (x @ np.asarray(w3, np.float64).T)
    else:
        if b1 is not None:
            a = a + np.asarray(b1, np.float64)[None, :]
        h = silu(a)
    h = round_to(dtype, h)
    y = h @ np.asarray(w2, np.float64).T
    if kind != SWIGLU and b2 is not None:
        y = y + np.asarray(b2, np.float64)[None, :]
    return h, round_f32(y)


def grouped_ffn(x_perm, offsets, p: dict, kind: int, dtype: int):
    """Every expert on its own rows of the expert-sorted buffer."""
    x_perm = np.asarray(x_perm)
    offsets = np.asarray(offsets, np.int64)
    n_experts = len(offsets) - 1
    d_ff = p["w1"].shape[1]
    d_model = p["w2"].shape[1]
    h = np.zeros((x_perm.shape[0], d_ff))
    y = np.zeros((x_perm.shape[0], d_model))
    for e in range(n_experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue        # empty expert batches are legal [DSEEK failure modes]
        h[lo:hi], y[lo:hi] = expert_ffn(
            x_perm[lo:hi], p["w1"][e], p["w2"][e], kind, dtype,
            w3=p["w3"][e] if kind == SWIGLU else None,
            b1=p["b1"][e] if p.get("b1") is not None else None,
            b2=p["b2"][e] if p.get("b2") is not None else None)
    return h, y


def shared_ffn(x, ws1, ws3, ws2, dtype: int) -> np.ndarray:
    """Always-on shared SwiGLU experts, each with weight 1, summed [DSEEK s.4].

    S[t] = sum_s W2_s (silu(W1_s x) * (W3_s x)), h rounded to the storage
    type, S kept unrounded (fp32 in the layer).
    """
    x = np.asarray(x, np.float64)
    out = np.zeros((x.shape[0], ws2.shape[1]))
    for s in range(ws1.shape[0]):
        h = silu(x @ np.asarray(ws1[s], np.float64).T) * (
            x @ np.asarray(ws3[s], np.float64).T)
        h = round_to(dtype, h)
        out += h @ np.asarray(ws2[s], np.float64).T
    return out


def combine(y_perm, row_of_slot, w, shared_out=None, n_tokens=None):
    """out[t] = sum_j w[t,j] * y[row_of_slot[t,j]] (+ S[t]); dropped slots add 0.

    The weighted scatter-add back to token order [QWEN index_add_; BUILD
    step 5; DSEEK s.3].  Float64, unrounded.
    """
    w = np.asarray(w, np.float64)
    n_tokens, k = w.shape
    y_perm = np.asarray(y_perm, np.float64)
    out = np.zeros((n_tokens, y_perm.shape[1]))
    rows = np.asarray(row_of_slot, np.int64).reshape(n_tokens, k)
    for j in range(k):
        r = rows[:, j]
        keep = r >= 0
        out[keep] += w[keep, j][:, None] * y_perm[r[keep]]
    if shared_out is not None:
        out += np.asarray(shared_out, np.float64)
    return out


def balance_statistic(counts, p, n_tokens: int, coef: float) -> float:
    """coef * sum_e frac_e * p_avg_e with frac_e = counts_e / N and
    p_avg_e = mean over tokens of p[t, e] [SER section 4]."""
    counts = np.asarray(counts, np.float64)
    frac = counts / float(n_tokens)
    p_avg = np.asarray(p, np.float64).sum(axis=0) / float(n_tokens)
    return float(coef * np.sum(frac * p_avg))


# --------------------------------------------------------------------------
# between steps: the selection-bias update and the load diagnostic
# --------------------------------------------------------------------------
def selection_bias_update(sel_bias, counts, gamma: float) -> np.ndarray:
    """b_e <- b_e + gamma * sign(mean load - load_e), in fp32.

    DSEEK s.2 adds a non-gradient balancing bias to the selection keys, and
    its study lab shows the per-expert load changing as that bias is
    updated; the pages do not state the update.  This is the plainest rule consistent
    with them (a reading, not a page's formula): an expert above the mean
    load is made less attractive by gamma, one below it more, one exactly
    at the mean is left alone.  The sign is decided on integers
    (E * load_e against the total) and the add is one fp32 add.
    """
    counts = np.asarray(counts, np.int64)
    b = np.asarray(sel_bias, np.float32)
    total = int(counts.sum())
    e = counts.shape[0]
    sign = np.sign(total - e * counts).astype(np.float32)   # +1 below the mean
    return (b + np.float32(gamma) * sign).astype(np.float32)


def load_cv(counts) -> float:
    """Coefficient of variation of the per-expert load: population standard
    deviation over the mean (DSEEK implementation plan, which asks for this
    statistic as a diagnostic of the load); 0 when nothing was routed."""
    c = np.asarray(counts, np.float64)
    m = c.mean() if c.size else 0.0
    if m == 0.0:
        return 0.0
    return float(np.sqrt(np.mean((c - m) ** 2)) / m)


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------
def forward(shape, values: dict) -> dict:
    """The sparse-MoE FFN forward of one workload, every stage returned.

    ``shape`` is any object with the workload fields (n_tokens, n_experts,
    top_k, expert, route, dtype, capacity_factor, n_shared, balance_coef);
    ``values`` holds the fp32 arrays the layer sees.  ``out`` is rounded to
    the layer's storage type; ``out_exact`` is the same sum before that last
    rounding.
    """
    x = values["x"]
    n_tokens = x.shape[0]
    logits = router_logits(x, values["w_router"], values.get("b_router"))
    idx, w, p = route(logits, shape.route, shape.top_k, values.get("sel_bias"))
    disp = dispatch(idx, shape.n_experts, shape.capacity_factor)
    x_perm = permute_rows(x, disp["token_of_row"])
    h, y = grouped_ffn(x_perm, disp["offsets"], values, shape.expert, shape.dtype)
    shared = None
    if shape.n_shared > 0:
        shared = round_f32(shared_ffn(x, values["ws1"], values["ws3"],
                                      values["ws2"], shape.dtype))
    out_exact = combine(y, disp["row_of_slot"], w, shared)
    out = round_to(shape.dtype, out_exact)
    bal = balance_statistic(disp["counts"], p, n_tokens, shape.balance_coef) \
        if n_tokens > 0 else 0.0
    res = dict(logits=logits, idx=idx, w=w, p=p, x_perm=x_perm, h=h, y=y,
               shared=shared, out=out, out_exact=out_exact, balance=bal)
    res.update(disp)
    return res


def forward_tokens(shape, values: dict, tokens) -> dict:
    """Output rows for a subset of tokens, computed one token at a time.

    Valid when no capacity limit applies (then a token's output depends on
    that token alone).  Used for sampled checks at full size.
    """
    if shape.capacity_factor and shape.capacity_factor > 0:
        raise ValueError("per-token outputs need a layer without capacity")
    tokens = np.asarray(tokens, np.int64)
    x = values["x"][tokens]
    logits = router_logits(x, values["w_router"], values.get("b_router"))
    idx, w, p = route(logits, shape.route, shape.top_k, values.get("sel_bias"))
    out = np.zeros((len(tokens), x.shape[1]))
    for i in range(len(tokens)):
        for j in range(shape.top_k):
            e = int(idx[i, j])
            _, y = expert_ffn(
                x[i:i + 1], values["w1"][e], values["w2"][e], shape.expert,
                shape.dtype,
                w3=values["w3"][e] if shape.expert == SWIGLU else None,
                b1=values["b1"][e] if values.get("b1") is not None else None,
                b2=values["b2"][e] if values.get("b2") is not None else None)
            out[i] += w[i, j] * y[0]
    if shape.n_shared > 0:
        out += round_f32(shared_ffn(x, values["ws1"], values["ws3"],
                                    values["ws2"], shape.dtype))
    return dict(logits=logits, idx=idx, w=w, out=round_to(shape.dtype, out),
                out_exact=out)
