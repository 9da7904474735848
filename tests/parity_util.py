"""Helpers shared by the GPU parity tests: uploads, tolerance checks and the
handling of routing near-ties.

Tolerances (stated by the layer's specification):
  * integer / index / byte results: bit-exact;
  * fp32 layer outputs: max |gpu - oracle| <= 1e-4 * RMS(oracle);
  * bf16 layer outputs (fp32 accumulation): max |gpu - oracle| <= 2e-2 * RMS(oracle);
  * the balance statistic: relative error <= 1e-4.
Layer outputs are compared with the oracle's value before its final storage
rounding: the tolerance bounds the computation, and a bf16 output may in
addition carry its own storage rounding, half a bf16 ulp of the value (no
bf16-output implementation can avoid that; the outputs here reach ~10x
their RMS, where half an ulp alone is ~3% of the RMS).  The hidden
activations h, which both sides round to bf16, may legitimately differ by
one bf16 ulp wherever the two unrounded values straddle a rounding
boundary, so they are checked element by element against one ulp.
"""
import functools

import numpy as np
import torch

from routing_dispatch_expert_05_b300 import moe as M
from routing_dispatch_expert_05_b300 import workloads as W

FP32_REL = 1e-4
BF16_REL = 2e-2
BALANCE_REL = 1e-4


def rel_tol(dtype):
    return BF16_REL if dtype == W.DTYPE_BF16 else FP32_REL


def assert_close_rms(got, ref, rel, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), what
    assert err <= rel * max(rms, 1e-30), f"{what}: max err {err:.3e} > {rel} * rms {rms:.3e}"


def assert_within_ulp(got, ref, dtype, what=""):
    """Element-wise: |gpu - oracle| <= one storage ulp of the oracle value
    (2^-7 relative for bf16) plus the fp32 accumulation bound (1e-4 of the
    RMS, which matters where a value is small after cancellation)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    assert np.isfinite(got).all(), what
    if dtype != W.DTYPE_BF16:
        assert_close_rms(got, ref, FP32_REL, what)
        return
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = 2.0 ** -7 * np.abs(ref) + FP32_REL * rms
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond one ulp, "
                           f"worst {float(np.max(np.abs(got - ref) - bound)):.3e}")
    # and the one-ulp differences are rare, not systematic
    assert np.mean(got != ref) < 0.02, f"{what}: {np.mean(got != ref):.3%} differ"


def half_ulp_bf16(a):
    """Half a bf16 unit in the last place of |a| (bf16 keeps 8 significant bits)."""
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def assert_output_close(got, exact, dtype, what=""):
    """Layer outputs: |gpu - exact| <= tol * RMS(exact) element by element,
    plus, for a bf16 output, half a bf16 ulp of the exact value."""
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    assert got.shape == exact.shape, (what, got.shape, exact.shape)
    if exact.size == 0:
        return
    assert np.isfinite(got).all(), what
    rms = float(np.sqrt(np.mean(exact ** 2)))
    tol = rel_tol(dtype) * max(rms, 1e-30)
    if dtype == W.DTYPE_BF16:
        bound = tol + half_ulp_bf16(exact)
    else:
        bound = tol + np.abs(exact) * 2.0 ** -24
    excess = np.abs(got - exact) - bound
    assert (excess <= 0).all(), (
        f"{what}: {int((excess > 0).sum())} outputs beyond tolerance, worst excess "
        f"{float(excess.max()):.3e} (rms {rms:.3e})")


def set_ambiguous_tokens(keys, k, margin):
    """Tokens whose selected SET depends on a gap below `margin` (the k-th and
    (k+1)-th best keys), and the experts such a near-tie may swap."""
    keys = np.asarray(keys, np.float64)
    n, e = keys.shape
    if k >= e:
        return np.zeros(n, bool), set()
    s = -np.sort(-keys, axis=1)
    amb = (s[:, k - 1] - s[:, k]) < margin
    experts = set()
    for t in np.nonzero(amb)[0]:
        lo, hi = s[t, k] - margin, s[t, k - 1] + margin
        experts.update(np.nonzero((keys[t] >= lo) & (keys[t] <= hi))[0].tolist())
    return amb, experts


def logit_margin(gpu_logits, oracle_logits):
    """Twice the largest logit difference (plus two fp32 ulps of the largest
    key): a gap in the oracle's keys wider than this decides the same
    ranking on both sides.  The sigmoid key's slope is at most 1/4, so the
    same margin covers it."""
    d = float(np.max(np.abs(np.asarray(gpu_logits, np.float64) -
                            np.asarray(oracle_logits, np.float64))))
    big = float(np.max(np.abs(oracle_logits))) if np.size(oracle_logits) else 0.0
    return 2.0 * d + 2.0 * big * 2.0 ** -23 + 1e-30


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.is_floating_point() \
        else t.detach().cpu().numpy()


def dev(a, dtype_code=W.DTYPE_F32):
    """numpy -> cuda tensor; float arrays become the layer dtype (exact for
    values already rounded to bf16)."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.is_floating_point():
        t = t.float()
        if dtype_code == W.DTYPE_BF16:
            t = t.to(torch.bfloat16)
    return t.cuda()


@functools.lru_cache(maxsize=None)
def _full_inputs(name):
    return W.make_inputs(W.WORKLOADS[name])


def inputs_for(name, n_tokens=None):
    """The workload's inputs, optionally restricted to its first n tokens
    (the same layer parameters either way)."""
    full = _full_inputs(name)
    return full if n_tokens is None else full.first_tokens(n_tokens)


def ambiguous_tokens(keys, k, margin):
    """Tokens whose ranking among the first k+1 keys is decided by a gap
    smaller than `margin` (where two correct implementations that differ by
    rounding may legitimately order experts differently)."""
    keys = np.asarray(keys, np.float64)
    n, e = keys.shape
    s = -np.sort(-keys, axis=1)
    upto = min(k + 1, e)
    if upto < 2:
        return np.zeros(n, bool)
    gaps = s[:, :upto - 1] - s[:, 1:upto]
    return (gaps < margin).any(axis=1)


def check_selection_valid(idx_gpu, keys, k, margin):
    """The chosen experts are distinct and every chosen key is within
    `margin` of the oracle's k-th best key."""
    keys = np.asarray(keys, np.float64)
    kth = -np.sort(-keys, axis=1)[:, k - 1]
    for t in range(idx_gpu.shape[0]):
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k
        assert (keys[t, sel] >= kth[t] - margin).all()


class Device:
    """Device copies of one workload's inputs plus a workspace."""

    def __init__(self, inputs: W.MoEInputs):
        self.inputs = inputs
        self.shape = inputs.shape
        self.cfg = M.make_config(self.shape)
        self.t = M.upload(inputs)
        self.weights = M.make_weights(self.t)
        self.ws = M.MoEWorkspace(self.cfg)
        self.tdtype = M.torch_dtype(self.shape.dtype)

    def empty(self, *shape, dtype=None):
        return torch.zeros(*shape, dtype=dtype or self.tdtype, device="cuda")

    def stats(self):
        E = self.shape.n_experts
        s = dict(counts=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                 kept=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                 dropped=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                 balance=torch.full((1,), -7.0, dtype=torch.float32, device="cuda"))
        return s, M.make_stats(**s)

    def device_error(self):
        return M.moe_read_device_error(self.ws)
