"""Python binding of the C ABI in ``include/moe.h`` (ctypes).

Argument marshalling only: every function here turns torch tensors into
device pointers, passes the current CUDA stream and raises ``MoEError`` on a
non-OK status.  All computation runs in ``libmoe_b300.so``; there is no CPU
path.  If the library has not been built, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = -1, -2, -3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_CHECK = -4, -5, -6
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
                -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_TIMEOUT",
                -6: "MOE_ERR_DEVICE_CHECK"}
MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTE_SOFTMAX_TOPK, MOE_ROUTE_TOPK_SOFTMAX, MOE_ROUTE_SIGMOID_BIAS = 0, 1, 2
MOE_EXPERT_SILU_MLP, MOE_EXPERT_SWIGLU = 0, 1

# every function include/moe.h declares (checked by the tests)
EXPORTED = ("moe_scratch_size", "moe_workspace_size", "moe_router_topk",
            "moe_route_logits", "moe_dispatch_permute",
            "moe_dispatch_permute_room", "moe_dispatch_permute_noalloc", "moe_expert_up",
            "moe_expert_up_gather", "moe_expert_down", "moe_grouped_ffn", "moe_shared_ffn", "moe_combine",
            "moe_forward", "moe_forward_timed", "moe_forward_host",
            "moe_update_selection_bias", "moe_backward_workspace_size", "moe_backward",
            "moe_check_grouping", "moe_check_wait_timeout", "moe_read_device_error",
            "moe_status_string", "moe_version")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class MoEConfig(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("d_ff_shared", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("route", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("balance_coef", ctypes.c_float)]


class MoEWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "b_router", "sel_bias", "w1", "b1", "w3", "w2", "b2",
                 "ws1", "ws3", "ws2")]


class MoEStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("counts", "kept", "dropped", "balance")]


class MoEGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("dx", "d_w_router", "d_b_router", "d_w1",
                                               "d_w3", "d_w2", "d_b1", "d_b2", "d_ws1",
                                               "d_ws3", "d_ws2")]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library once; raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing "
            "(run `python -m routing_dispatch_expert_05_b300.build`)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    cfgp, wp, sp = P(MoEConfig), P(MoEWeights), P(MoEStats)
    sig = {
        "moe_scratch_size": [cfgp, P(sz)],
        "moe_workspace_size": [cfgp, P(sz)],
        "moe_router_topk": [cfgp, vp, wp, vp, vp, vp, sp, vp, sz, vp],
        "moe_route_logits": [cfgp, vp, vp, vp, vp, sp, vp, sz, vp],
        "moe_dispatch_permute": [cfgp, vp, vp, vp, vp, vp, vp, sp, vp, sz, vp],
        "moe_dispatch_permute_noalloc": [cfgp, vp, vp, vp, vp, vp, vp, sp, vp],
        "moe_dispatch_permute_room": [cfgp, vp, vp, vp, vp, vp, vp, vp, sp, vp, sz, vp],
        "moe_expert_up": [cfgp, vp, vp, wp, vp, vp, sz, vp],
        "moe_expert_up_gather": [cfgp, vp, vp, vp, wp, vp, vp, sz, vp],
        "moe_expert_down": [cfgp, vp, vp, wp, vp, vp, sz, vp],
        "moe_grouped_ffn": [cfgp, vp, vp, wp, vp, vp, vp, sz, vp],
        "moe_shared_ffn": [cfgp, vp, wp, vp, vp, vp, sz, vp],
        "moe_combine": [cfgp, vp, vp, vp, vp, vp, vp, sz, vp],
        "moe_forward": [cfgp, vp, wp, vp, sp, vp, sz, vp],
        "moe_forward_host": [cfgp, vp, wp, vp, sp, vp, sz, vp],
        "moe_forward_timed": [cfgp, vp, wp, vp, sp, vp, sz, vp, P(vp), ctypes.c_int32],
        "moe_read_device_error": [vp, P(ctypes.c_int32), vp],
        "moe_update_selection_bias": [cfgp, vp, vp, ctypes.c_float, vp, vp],
        "moe_backward_workspace_size": [cfgp, P(sz)],
        "moe_check_wait_timeout": [vp, sz, ctypes.c_int64, vp],
        "moe_check_grouping": [cfgp, vp, vp, vp, vp, vp, sz, vp],
        "moe_backward": [cfgp, vp, wp, vp, ctypes.c_float, P(MoEGrads), vp, sz, vp],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int32
    lib.moe_status_string.argtypes = [ctypes.c_int32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_version.argtypes = []
    lib.moe_version.restype = ctypes.c_int32
    _lib = lib
    return lib


# ---------------------------------------------------------------- helpers
def ptr(t) -> Optional[int]:
    """Device (or host) address of a tensor; None for None; ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "tensor"):        # MoEWorkspace
        t = t.tensor
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where)


def make_config(shape, n_tokens: Optional[int] = None) -> MoEConfig:
    """moe_config_t from a workload description (fields as in workloads.MoEShape)."""
    return MoEConfig(
        n_tokens=shape.n_tokens if n_tokens is None else n_tokens,
        d_model=shape.d_model, n_experts=shape.n_experts, top_k=shape.top_k,
        d_ff=shape.d_ff, n_shared=shape.n_shared, d_ff_shared=shape.d_ff_shared,
        capacity_factor=shape.capacity_factor, route=shape.route,
        expert=shape.expert, dtype=shape.dtype, has_bias=int(shape.has_bias),
        balance_coef=shape.balance_coef)


def make_weights(tensors: Dict[str, torch.Tensor]) -> MoEWeights:
    w = MoEWeights()
    for name, _ in MoEWeights._fields_:
        setattr(w, name, ptr(tensors.get(name)))
    return w


def make_stats(counts=None, kept=None, dropped=None, balance=None) -> MoEStats:
    return MoEStats(ptr(counts), ptr(kept), ptr(dropped), ptr(balance))


def scratch_size(cfg: MoEConfig) -> int:
    n = ctypes.c_size_t()
    _check(load_library().moe_scratch_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_scratch_size")
    return n.value


def workspace_size(cfg: MoEConfig) -> int:
    n = ctypes.c_size_t()
    _check(load_library().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_workspace_size")
    return n.value


def _rows_arg(t, cfg, name):
    """A token-row argument ([n_tokens, d_model] in the layer dtype) as an
    address.  A tensor smaller than the config declares is refused here: the
    library takes plain pointers and would read or write past its end."""
    if isinstance(t, torch.Tensor):
        es = 2 if cfg.dtype == MOE_BF16 else 4
        need = int(cfg.n_tokens) * int(cfg.d_model) * es
        have = t.numel() * t.element_size()
        if have < need:
            raise ValueError(f"{name}: {have} bytes, the config needs {need} "
                             f"({cfg.n_tokens} tokens x {cfg.d_model})")
    return ptr(t)


def _ws(ws):
    if ws is None:
        return None, 0
    if hasattr(ws, "tensor"):
        ws = ws.tensor
    return ptr(ws), ws.numel() * ws.element_size()


# ---------------------------------------------------------------- stages
def moe_router_topk(cfg, x, weights: MoEWeights, logits, idx, w, stats, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_router_topk(
        ctypes.byref(cfg), _rows_arg(x, cfg, "x"), ctypes.byref(weights), ptr(logits),
        ptr(idx),
        ptr(w), ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_router_topk")


def moe_route_logits(cfg, logits, sel_bias, idx, w, stats, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_route_logits(
        ctypes.byref(cfg), ptr(logits), ptr(sel_bias), ptr(idx), ptr(w),
        ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_route_logits")


def moe_dispatch_permute(cfg, idx, x, offsets, row_of_slot, token_of_row, x_perm,
                         stats, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_dispatch_permute(
        ctypes.byref(cfg), ptr(idx), _rows_arg(x, cfg, "x"), ptr(offsets), ptr(row_of_slot),
        ptr(token_of_row), ptr(x_perm),
        ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_dispatch_permute")


def moe_dispatch_permute_room(cfg, idx, x, room, offsets, row_of_slot, token_of_row,
                              x_perm, stats, ws, stream=None):
    """moe_dispatch_permute with a per-expert capacity room [E] (int32)."""
    wp, wb = _ws(ws)
    _check(load_library().moe_dispatch_permute_room(
        ctypes.byref(cfg), ptr(idx), _rows_arg(x, cfg, "x"), ptr(room), ptr(offsets),
        ptr(row_of_slot),
        ptr(token_of_row), ptr(x_perm),
        ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_dispatch_permute_room")


def moe_dispatch_permute_noalloc(cfg, idx, x, offsets, row_of_slot, token_of_row,
                                 x_perm, stats, stream=None):
    """moe_dispatch_permute without a workspace, for callers that cannot give
    the library device memory (its scratch is a fixed array in the library:
    n_tokens <= 65536; overlapping calls race)."""
    _check(load_library().moe_dispatch_permute_noalloc(
        ctypes.byref(cfg), ptr(idx), _rows_arg(x, cfg, "x"), ptr(offsets), ptr(row_of_slot),
        ptr(token_of_row), ptr(x_perm),
        ctypes.byref(stats) if stats is not None else None, _stream(stream)),
        "moe_dispatch_permute_noalloc")


def moe_expert_up(cfg, x_perm, offsets, weights: MoEWeights, h, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_expert_up(
        ctypes.byref(cfg), ptr(x_perm), ptr(offsets), ctypes.byref(weights), ptr(h),
        wp, wb, _stream(stream)), "moe_expert_up")


def moe_expert_up_gather(cfg, x, token_of_row, offsets, weights: MoEWeights, h, ws,
                         stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_expert_up_gather(
        ctypes.byref(cfg), _rows_arg(x, cfg, "x"), ptr(token_of_row), ptr(offsets),
        ctypes.byref(weights), ptr(h), wp, wb, _stream(stream)), "moe_expert_up_gather")


def moe_expert_down(cfg, h, offsets, weights: MoEWeights, y, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_expert_down(
        ctypes.byref(cfg), ptr(h), ptr(offsets), ctypes.byref(weights), ptr(y),
        wp, wb, _stream(stream)), "moe_expert_down")


def moe_grouped_ffn(cfg, x_perm, offsets, weights: MoEWeights, h, y, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_grouped_ffn(
        ctypes.byref(cfg), ptr(x_perm), ptr(offsets), ctypes.byref(weights), ptr(h),
        ptr(y), wp, wb, _stream(stream)), "moe_grouped_ffn")


def moe_shared_ffn(cfg, x, weights: MoEWeights, h_shared, shared_out, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_shared_ffn(
        ctypes.byref(cfg), _rows_arg(x, cfg, "x"), ctypes.byref(weights), ptr(h_shared),
        ptr(shared_out), wp, wb, _stream(stream)), "moe_shared_ffn")


def moe_combine(cfg, y, row_of_slot, w, shared_out, out, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_combine(
        ctypes.byref(cfg), ptr(y), ptr(row_of_slot), ptr(w), ptr(shared_out),
        _rows_arg(out, cfg, "out"), wp, wb, _stream(stream)), "moe_combine")


def moe_forward(cfg, x, weights: MoEWeights, out, stats, ws, stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_forward(
        ctypes.byref(cfg), _rows_arg(x, cfg, "x"), ctypes.byref(weights),
        _rows_arg(out, cfg, "out"),
        ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_forward")


FORWARD_STAGES = ("router", "dispatch", "expert_up", "expert_down", "shared", "combine")
MOE_FORWARD_EVENTS = len(FORWARD_STAGES) + 1


def moe_forward_timed(cfg, x, weights: MoEWeights, out, stats, ws, events, stream=None):
    """moe_forward recording ``events`` (MOE_FORWARD_EVENTS torch.cuda.Event
    objects with timing enabled): before the layer and after each stage in
    FORWARD_STAGES."""
    if len(events) != MOE_FORWARD_EVENTS:
        raise ValueError(f"need {MOE_FORWARD_EVENTS} events")
    handles = []
    for ev in events:
        if not ev.cuda_event:            # torch creates the CUDA event lazily
            ev.record()
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles)
    wp, wb = _ws(ws)
    _check(load_library().moe_forward_timed(
        ctypes.byref(cfg), _rows_arg(x, cfg, "x"), ctypes.byref(weights),
        _rows_arg(out, cfg, "out"),
        ctypes.byref(stats) if stats is not None else None, wp, wb, _stream(stream),
        arr, len(handles)), "moe_forward_timed")


def moe_forward_host(cfg, x_host, weights: MoEWeights, out_host, stats, ws,
                     stream=None):
    wp, wb = _ws(ws)
    _check(load_library().moe_forward_host(
        ctypes.byref(cfg), _rows_arg(x_host, cfg, "x_host"), ctypes.byref(weights),
        _rows_arg(out_host, cfg, "out_host"),
        ctypes.byref(stats) if stats is not None else None, wp, wb,
        _stream(stream)), "moe_forward_host")


def backward_workspace_size(cfg: MoEConfig) -> int:
    n = ctypes.c_size_t()
    _check(load_library().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def make_grads(dx, d_w_router, d_w1, d_w2, d_w3=None, d_b_router=None, d_b1=None,
               d_b2=None, d_ws1=None, d_ws3=None, d_ws2=None) -> MoEGrads:
    return MoEGrads(ptr(dx), ptr(d_w_router), ptr(d_b_router), ptr(d_w1), ptr(d_w3),
                    ptr(d_w2), ptr(d_b1), ptr(d_b2), ptr(d_ws1), ptr(d_ws3), ptr(d_ws2))


def moe_backward(cfg, x, weights: MoEWeights, dout, d_balance, grads: MoEGrads, ws,
                 stream=None):
    """Gradients of <dout, out> + d_balance * balance (routing held fixed)
    into the fp32 arrays of `grads`; ws holds backward_workspace_size bytes."""
    wp, wb = _ws(ws)
    _check(load_library().moe_backward(ctypes.byref(cfg), _rows_arg(x, cfg, "x"),
                                       ctypes.byref(weights), _rows_arg(dout, cfg, "dout"),
                                       float(d_balance), ctypes.byref(grads), wp, wb,
                                       _stream(stream)), "moe_backward")


def moe_update_selection_bias(cfg, counts, sel_bias, gamma, load_cv=None, stream=None):
    """sel_bias += gamma * sign(mean load - counts) (in place) and the load's
    coefficient of variation into load_cv; both tensors may be None (not
    both)."""
    _check(load_library().moe_update_selection_bias(
        ctypes.byref(cfg), ptr(counts), ptr(sel_bias), float(gamma), ptr(load_cv),
        _stream(stream)), "moe_update_selection_bias")


def moe_check_grouping(cfg, idx, offsets, row_of_slot, token_of_row, ws, stream=None):
    """Check a grouping on the device; a failure shows in the error word."""
    wp, wb = _ws(ws)
    _check(load_library().moe_check_grouping(
        ctypes.byref(cfg), ptr(idx), ptr(offsets), ptr(row_of_slot), ptr(token_of_row),
        wp, wb, _stream(stream)), "moe_check_grouping")


def moe_check_wait_timeout(ws, limit_ns: int, stream=None):
    """Run the GEMMs' bounded wait out on purpose (see moe.h)."""
    wp, wb = _ws(ws)
    _check(load_library().moe_check_wait_timeout(wp, wb, int(limit_ns), _stream(stream)),
           "moe_check_wait_timeout")


def moe_read_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32()
    _check(load_library().moe_read_device_error(ptr(ws), ctypes.byref(code),
                                                _stream(stream)),
           "moe_read_device_error")
    return code.value


def status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


# ------------------------------------------------------ device residency
def torch_dtype(dtype_code: int):
    return torch.bfloat16 if dtype_code == MOE_BF16 else torch.float32


def upload(inputs, device="cuda") -> Dict[str, torch.Tensor]:
    """Copy a workloads.MoEInputs to device tensors in the layer dtype.

    bf16 tensors are uploaded from their exact bit patterns.
    """
    out = {}
    for name in inputs.values:
        if name in inputs.bits:
            t = torch.from_numpy(inputs.bits[name].view("int16").copy())
            out[name] = t.to(device).view(torch.bfloat16)
        else:
            out[name] = torch.from_numpy(inputs.values[name].copy()).to(device)
    return out


class MoEWorkspace:
    """A zero-filled workspace for moe_forward of one configuration."""

    def __init__(self, cfg: MoEConfig, device="cuda", forward: bool = True,
                 backward: bool = False):
        n = backward_workspace_size(cfg) if backward else (
            workspace_size(cfg) if forward else scratch_size(cfg))
        self.tensor = torch.zeros(max(n, 256), dtype=torch.uint8, device=device)

    @property
    def nbytes(self) -> int:
        return self.tensor.numel()

    def reset(self) -> None:
        """Zero the workspace again, on the current stream.  Needed only after
        a call returned MOE_ERR_CUDA, which can leave the running selection
        totals or the device error word set; every other call leaves the
        workspace ready for the next."""
        self.tensor.zero_()
