"""Seeded synthetic workloads for the sparse-MoE FFN forward.

This module only draws random inputs and describes the five workload shapes;
it holds none of the layer's arithmetic (no router, no selection, no
dispatch, no FFN, no combine).  Both the CUDA path's tests/benchmark and the
CPU oracle are fed from here, so the module deliberately imports neither.

The shapes follow the pages' workloads:

* ``toy_top2_fp32`` -- the 8-expert top-2 toy of "Tutorial -- MoE SER Expert
  Routing" (section 1 configuration: input 64, expert 128, output 64;
  section 2 input ``(4, 16, 64)``), with SiLU-MLP experts as in "Expert
  Networks > Code Implementation" (In[7]).
* ``capacity_top2_fp32`` / ``capacity_top2_bf16`` -- the capacity-constrained
  8-expert setting of "Expert Networks > Code Implementation" (In[7]: d_model
  256, d_ff 512, biases; In[10]: capacity from capacity_factor 1.25), scaled
  to 4096 tokens with top-2 routing and a skewing per-expert logit offset.
* ``deepseek_v3_block`` -- "DeepSeek 5.7: MoE from scratch" sections 1-4:
  SwiGLU experts, sigmoid affinities plus a selection-only balancing bias,
  two always-on shared experts.
* ``qwen3_moe`` -- the Qwen3 ``MoEFeedForward`` described on
  "Implementing Mixed Expert (MoE) layers" (Core Algorithmic Steps): topk on
  raw gate logits, softmax over the k, SwiGLU experts without bias; 128
  experts, d_ff 768, with a Zipf-skewed per-expert logit offset.
* ``decode_stream`` -- 64 tokens through the same 128-expert geometry: a
  weight-streaming (decode-shaped) case.

Randomness: NumPy ``default_rng(seed)`` (PCG64).  Values are drawn in fp32 and,
for bf16 workloads, rounded to bf16 (round to nearest even) before either side
sees them, so both sides start from identical bit patterns.  Draw order: the
expert stacks W1 (gate), b1, W3 (up), W2 (down), b2, the shared stacks, the
router weight, the router bias (or logit offset), the selection bias, and x
last -- so the layer's parameters do not depend on the number of tokens, and
the two 128-expert workloads (same seed) share their expert weights.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

ROUTE_SOFTMAX_TOPK = 0   # softmax over all E, select top-k, renormalise
ROUTE_TOPK_SOFTMAX = 1   # select top-k raw logits, softmax over the k
ROUTE_SIGMOID_BIAS = 2   # select on sigmoid(l)+b, weight = sigmoid(l)/sum_sel
EXPERT_SILU_MLP = 0      # w2 silu(w1 x + b1) + b2
EXPERT_SWIGLU = 1        # w2 (silu(w1 x) * (w3 x))
DTYPE_F32 = 0
DTYPE_BF16 = 1


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """One workload: layer geometry, routing mode, precision and seed."""
    name: str
    n_tokens: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    expert: int
    route: int
    dtype: int
    has_bias: bool = False          # expert biases b1 [E,F], b2 [E,d]
    router_bias: str = "none"       # "none" | "normal" | "offset_normal" | "zipf"
    router_offset_std: float = 0.0  # std of the per-expert offset ("offset_normal")
    zipf_s: float = 0.0             # exponent of the Zipf offset ("zipf")
    sel_bias_range: float = 0.0     # U(-r, r) selection bias (sigmoid mode)
    capacity_factor: float = 0.0    # <= 0: no capacity limit
    n_shared: int = 0
    d_ff_shared: int = 0
    balance_coef: float = 0.01
    seed: int = 0

    @property
    def assignments(self) -> int:
        return self.n_tokens * self.top_k

    def replace(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, MoEShape] = {
    "toy_top2_fp32": MoEShape(
        name="toy_top2_fp32", n_tokens=64, d_model=64, n_experts=8, top_k=2,
        d_ff=128, expert=EXPERT_SILU_MLP, route=ROUTE_SOFTMAX_TOPK,
        dtype=DTYPE_F32, has_bias=True, router_bias="normal", seed=0),
    "capacity_top2_fp32": MoEShape(
        name="capacity_top2_fp32", n_tokens=4096, d_model=256, n_experts=8,
        top_k=2, d_ff=512, expert=EXPERT_SILU_MLP, route=ROUTE_SOFTMAX_TOPK,
        dtype=DTYPE_F32, has_bias=True, router_bias="offset_normal",
        router_offset_std=1.5, capacity_factor=1.25, seed=2),
    "capacity_top2_bf16": MoEShape(
        name="capacity_top2_bf16", n_tokens=4096, d_model=256, n_experts=8,
        top_k=2, d_ff=512, expert=EXPERT_SILU_MLP, route=ROUTE_SOFTMAX_TOPK,
        dtype=DTYPE_BF16, has_bias=True, router_bias="offset_normal",
        router_offset_std=1.5, capacity_factor=1.25, seed=2),
    "deepseek_v3_block": MoEShape(
        name="deepseek_v3_block", n_tokens=8192, d_model=2048, n_experts=64,
        top_k=6, d_ff=1024, expert=EXPERT_SWIGLU, route=ROUTE_SIGMOID_BIAS,
        dtype=DTYPE_BF16, sel_bias_range=0.1, n_shared=2, d_ff_shared=1024,
        seed=3),
    "qwen3_moe": MoEShape(
        name="qwen3_moe", n_tokens=16384, d_model=2048, n_experts=128,
        top_k=8, d_ff=768, expert=EXPERT_SWIGLU, route=ROUTE_TOPK_SOFTMAX,
        dtype=DTYPE_BF16, router_bias="zipf", zipf_s=1.1, seed=4),
    "decode_stream": MoEShape(
        name="decode_stream", n_tokens=64, d_model=2048, n_experts=128,
        top_k=8, d_ff=768, expert=EXPERT_SWIGLU, route=ROUTE_TOPK_SOFTMAX,
        dtype=DTYPE_BF16, seed=4),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round to nearest even.

    Finite values and infinities only (no NaN is ever drawn): the rounding
    increment then never carries out of 32 bits, so the sum stays uint32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u >> 16) & 1
    r += 0x7FFF
    r += u
    r >>= 16
    return r.astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> the fp32 values they represent."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, std):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


@dataclasses.dataclass
class MoEInputs:
    """Host arrays for one workload.

    ``values[name]`` is the fp32 array of what the layer sees (already
    bf16-rounded for bf16 workloads); ``bits[name]`` is the uint16 bf16 bit
    pattern (bf16 workloads only) for upload.  Weight layout is the PyTorch
    Linear layout ``[out, in]`` stacked over experts.
    """
    shape: MoEShape
    values: Dict[str, np.ndarray]
    bits: Dict[str, np.ndarray]

    def first_tokens(self, n: int) -> "MoEInputs":
        """The same layer applied to the first n tokens only (views, no copy)."""
        have = self.values["x"].shape[0]
        if not 0 <= n <= have:
            raise ValueError(f"first_tokens({n}): these inputs hold {have} tokens")
        v = dict(self.values)
        b = dict(self.bits)
        v["x"] = self.values["x"][:n]
        if "x" in b:
            b["x"] = self.bits["x"][:n]
        return MoEInputs(shape=self.shape.replace(n_tokens=n), values=v, bits=b)

    def device_array(self, name: str) -> np.ndarray:
        """The array to upload: bf16 bits for bf16 parameters, fp32 otherwise."""
        if name in self.bits:
            return self.bits[name]
        return self.values[name]


# names of tensors stored in the layer dtype (sel_bias is always fp32)
PARAM_NAMES = ("x", "w_router", "b_router", "w1", "b1", "w3", "w2", "b2",
               "ws1", "ws3", "ws2")


def make_inputs(shape: MoEShape, seed: Optional[int] = None,
                n_tokens: Optional[int] = None) -> MoEInputs:
    """Draw the seeded inputs of ``shape`` (optionally overriding seed / N)."""
    s = shape if n_tokens is None else shape.replace(n_tokens=n_tokens)
    rng = np.random.default_rng(s.seed if seed is None else seed)
    N, d, E, F = s.n_tokens, s.d_model, s.n_experts, s.d_ff
    v: Dict[str, np.ndarray] = {}
    v["w1"] = _normal(rng, (E, F, d), 1.0 / math.sqrt(d))
    if s.has_bias:
        v["b1"] = _normal(rng, (E, F), 1.0 / math.sqrt(d))
    if s.expert == EXPERT_SWIGLU:
        v["w3"] = _normal(rng, (E, F, d), 1.0 / math.sqrt(d))
    v["w2"] = _normal(rng, (E, d, F), 1.0 / math.sqrt(F))
    if s.has_bias:
        v["b2"] = _normal(rng, (E, d), 1.0 / math.sqrt(F))
    if s.n_shared > 0:
        S, Fs = s.n_shared, s.d_ff_shared
        v["ws1"] = _normal(rng, (S, Fs, d), 1.0 / math.sqrt(d))
        v["ws3"] = _normal(rng, (S, Fs, d), 1.0 / math.sqrt(d))
        v["ws2"] = _normal(rng, (S, d, Fs), 1.0 / math.sqrt(Fs))
    v["w_router"] = _normal(rng, (E, d), 1.0 / math.sqrt(d))
    if s.router_bias == "normal":
        v["b_router"] = _normal(rng, (E,), 1.0 / math.sqrt(d))
    elif s.router_bias == "offset_normal":
        v["b_router"] = _normal(rng, (E,), s.router_offset_std)
    elif s.router_bias == "zipf":
        rank = rng.permutation(E).astype(np.float64) + 1.0
        v["b_router"] = (-s.zipf_s * np.log(rank)).astype(np.float32)
    if s.route == ROUTE_SIGMOID_BIAS:
        r = s.sel_bias_range
        v["sel_bias"] = rng.uniform(-r, r, size=(E,)).astype(np.float32)
    v["x"] = _normal(rng, (N, d), 1.0)
    bits: Dict[str, np.ndarray] = {}
    if s.dtype == DTYPE_BF16:
        for name in PARAM_NAMES:
            if name in v:
                bits[name] = bf16_bits(v[name])
                v[name] = bits_to_f32(bits[name])
    return MoEInputs(shape=s, values=v, bits=bits)


def make_logits(n_tokens: int, n_experts: int, seed: int,
                kind: str = "normal") -> np.ndarray:
    """Seeded fp32 router logits fed identically to both sides.

    ``normal``: N(0,1).  ``ties``: small integers in {-2..2} (forces exact
    ties).  ``signed_zero``: mixes +0.0 and -0.0 with a few nonzero values,
    so -0 == +0 ties are exercised.
    """
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((n_tokens, n_experts), dtype=np.float32)
    if kind == "ties":
        return rng.integers(-2, 3, size=(n_tokens, n_experts)).astype(np.float32)
    if kind == "signed_zero":
        z = np.where(rng.random((n_tokens, n_experts)) < 0.5, 0.0, -0.0)
        z = z.astype(np.float32)
        hot = rng.random((n_tokens, n_experts)) < 0.1
        z[hot] = rng.integers(-1, 2, size=int(hot.sum())).astype(np.float32)
        return z
    raise ValueError(kind)


def make_assignments(n_tokens: int, n_experts: int, top_k: int, seed: int,
                     zipf_s: float = 0.0) -> np.ndarray:
    """Seeded routing indices idx[N,k]: k distinct experts per token.

    With ``zipf_s > 0`` expert e is drawn with probability proportional to
    (e+1)^-s, giving a heavily skewed load (many empty experts for large E).
    """
    rng = np.random.default_rng(seed)
    if zipf_s > 0:
        pr = (np.arange(1, n_experts + 1, dtype=np.float64)) ** (-zipf_s)
        pr /= pr.sum()
    else:
        pr = None
    idx = np.empty((n_tokens, top_k), dtype=np.int32)
    for t in range(n_tokens):
        idx[t] = rng.choice(n_experts, size=top_k, replace=False, p=pr)
    return idx
