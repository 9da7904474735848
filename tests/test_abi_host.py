"""The C-ABI library loads, exports every function include/moe.h declares,
and rejects invalid arguments on the host -- no GPU needed (no call here
reaches the device)."""
import ctypes
import os
import re

import pytest

from routing_dispatch_expert_05_b300 import build as B
from routing_dispatch_expert_05_b300 import moe as M
from routing_dispatch_expert_05_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_binding_functions():
    assert _declared_functions() == sorted(M.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.moe_version() >= 100
    for code in M.STATUS_NAMES:
        assert lib.moe_status_string(code).decode()
    assert lib.moe_status_string(12345).decode() == "unknown status"


def test_config_struct_layout_matches_header():
    # int64 + 6 int32 + float + 4 int32 + float = 8 + 24 + 4 + 16 + 4 = 56
    assert ctypes.sizeof(M.MoEConfig) == 56
    assert ctypes.sizeof(M.MoEWeights) == 11 * 8
    assert ctypes.sizeof(M.MoEStats) == 4 * 8


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workspace_sizes_cover_the_intermediates(lib, name):
    shape = W.WORKLOADS[name]
    cfg = M.make_config(shape)
    scratch = M.scratch_size(cfg)
    total = M.workspace_size(cfg)
    es = 2 if shape.dtype == W.DTYPE_BF16 else 4
    nk = shape.n_tokens * shape.top_k
    # the forward keeps x_perm [N*k, d] and h [N*k, F] in the layer dtype and
    # the expert outputs y [N*k, d] in at least 16 bits
    floor = nk * (shape.d_model + shape.d_ff) * es + nk * shape.d_model * 2
    assert scratch >= shape.n_tokens * shape.n_experts * 4
    assert total >= scratch + floor


def _bad(**kw):
    base = dict(W.WORKLOADS["toy_top2_fp32"].__dict__)
    base.update(kw)
    return M.make_config(W.MoEShape(**base))


@pytest.mark.parametrize("kw", [
    dict(top_k=0), dict(top_k=9), dict(n_experts=0), dict(n_experts=300),
    dict(d_model=0), dict(d_model=66), dict(d_ff=130), dict(dtype=5),
    dict(route=3), dict(expert=2), dict(n_tokens=-1), dict(n_shared=-1),
    dict(n_shared=1, d_ff_shared=0), dict(expert=W.EXPERT_SWIGLU, has_bias=True),
    dict(capacity_factor=float("nan"))])
def test_invalid_config_rejected(lib, kw):
    cfg = _bad(**kw)
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == -1


def test_bf16_needs_multiple_of_8(lib):
    cfg = _bad(dtype=W.DTYPE_BF16, d_model=68)   # 68 % 8 != 0
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == -1


def test_too_many_assignments_unsupported(lib):
    cfg = _bad(n_tokens=2 ** 31, top_k=2)
    n = ctypes.c_size_t()
    assert lib.moe_scratch_size(ctypes.byref(cfg), ctypes.byref(n)) == -2


def test_stage_calls_reject_bad_pointers_before_the_device(lib):
    cfg = M.make_config(W.WORKLOADS["toy_top2_fp32"])
    w = M.MoEWeights()
    buf = ctypes.create_string_buffer(1 << 20)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    # missing router weight
    st = lib.moe_router_topk(ctypes.byref(cfg), addr, ctypes.byref(w), None, addr,
                             addr, None, addr, 1 << 19, None)
    assert st == -1
    # misaligned x
    w.w_router = addr
    st = lib.moe_router_topk(ctypes.byref(cfg), addr + 4, ctypes.byref(w), None,
                             addr, addr, None, addr, 1 << 19, None)
    assert st == -1
    # workspace too small
    st = lib.moe_router_topk(ctypes.byref(cfg), addr, ctypes.byref(w), None, addr,
                             addr, None, addr, 16, None)
    assert st == -3
    # sigmoid mode without the selection bias
    cfg2 = _bad(route=W.ROUTE_SIGMOID_BIAS)
    st = lib.moe_route_logits(ctypes.byref(cfg2), addr, None, addr, addr, None,
                              addr, 1 << 19, None)
    assert st == -1
    # shared experts requested but absent
    st = lib.moe_shared_ffn(ctypes.byref(cfg), addr, ctypes.byref(w), addr, addr,
                            addr, 1 << 19, None)
    assert st == -1
    # forward with a SwiGLU layer but no up projection
    cfg3 = _bad(expert=W.EXPERT_SWIGLU, has_bias=False)
    w.w1 = addr
    w.w2 = addr
    st = lib.moe_forward(ctypes.byref(cfg3), addr, ctypes.byref(w), addr, None,
                         addr, 1 << 40, None)
    assert st == -1


def test_binding_refuses_token_rows_smaller_than_the_config(lib):
    """The Python binding checks each [n_tokens, d_model] tensor against the
    config before the call: the library takes plain pointers and would read
    (or write) past the end of a shorter buffer."""
    import torch
    shape = W.WORKLOADS["capacity_top2_bf16"]
    cfg = M.make_config(shape)
    short = torch.zeros(shape.n_tokens - 1, shape.d_model, dtype=torch.bfloat16)
    full = torch.zeros(shape.n_tokens, shape.d_model, dtype=torch.bfloat16)
    w = M.MoEWeights()
    sts = None
    with pytest.raises(ValueError, match="x:"):
        M.moe_forward(cfg, short, w, full, sts, None)
    with pytest.raises(ValueError, match="out:"):
        M.moe_forward(cfg, full, w, short, sts, None)
    with pytest.raises(ValueError, match="x_host:"):
        M.moe_forward_host(cfg, short, w, full, sts, None)
    with pytest.raises(ValueError, match="x:"):
        M.moe_router_topk(cfg, short, w, None, None, None, None, None)
    with pytest.raises(ValueError, match="x:"):
        M.moe_dispatch_permute(cfg, None, short, None, None, None, None, None, None)
    with pytest.raises(ValueError, match="out:"):
        M.moe_combine(cfg, None, None, None, None, short, None)
    with pytest.raises(ValueError, match="dout:"):
        M.moe_backward(cfg, full, w, short, 0.0, M.MoEGrads(), None)
    # big enough: the call reaches the library, which rejects the missing
    # workspace on the host
    with pytest.raises(M.MoEError):
        M.moe_forward(cfg, full, w, full, sts, None)


def test_forward_timed_rejects_a_wrong_event_count(lib):
    cfg = M.make_config(W.WORKLOADS["toy_top2_fp32"])
    w = M.MoEWeights()
    evs = (ctypes.c_void_p * 3)(1, 2, 3)
    st = lib.moe_forward_timed(ctypes.byref(cfg), None, ctypes.byref(w), None, None,
                               None, 0, None, evs, 3)
    assert st == M.MOE_ERR_INVALID_ARG
    st = lib.moe_forward_timed(ctypes.byref(cfg), None, ctypes.byref(w), None, None,
                               None, 0, None, None, M.MOE_FORWARD_EVENTS)
    assert st == M.MOE_ERR_INVALID_ARG


def test_bias_update_rejects_bad_arguments(lib):
    cfg = M.make_config(W.WORKLOADS["toy_top2_fp32"])
    buf = ctypes.create_string_buffer(4096)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    f = lib.moe_update_selection_bias
    assert f(ctypes.byref(cfg), None, addr, 1e-3, addr, None) == M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(cfg), addr, None, 1e-3, None, None) == M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(cfg), addr, addr, float("nan"), addr, None) == M.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(cfg), addr, addr + 2, 1e-3, None, None) == M.MOE_ERR_INVALID_ARG
    bad = _bad(n_experts=0)
    assert f(ctypes.byref(bad), addr, addr, 1e-3, addr, None) == M.MOE_ERR_INVALID_ARG


def test_backward_rejects_unsupported_layers(lib):
    """fp32 layers and widths the tensor-core backward does not tile (d, F or
    Fs not a multiple of 64, E not a multiple of 8) get MOE_ERR_UNSUPPORTED
    before anything is enqueued; a supported layer with a gradient output
    missing (d_w3 of SwiGLU, d_b1 / d_b2 with expert biases, the shared
    experts' gradients) gets MOE_ERR_INVALID_ARG (no GPU needed)."""
    buf = ctypes.create_string_buffer(4096)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    w = M.MoEWeights()
    g = M.MoEGrads()
    bf = W.WORKLOADS["capacity_top2_bf16"]
    for shape in (W.WORKLOADS["toy_top2_fp32"], bf.replace(d_model=72),
                  bf.replace(d_ff=96), bf.replace(n_experts=4),
                  W.WORKLOADS["deepseek_v3_block"].replace(d_ff_shared=96)):
        cfg = M.make_config(shape)
        st = lib.moe_backward(ctypes.byref(cfg), addr, ctypes.byref(w), addr, 0.0,
                              ctypes.byref(g), addr, 1 << 20, None)
        assert st == M.MOE_ERR_UNSUPPORTED, shape
    full = dict(dx=addr, d_w_router=addr, d_w1=addr, d_w3=addr, d_w2=addr, d_b1=addr,
                d_b2=addr, d_ws1=addr, d_ws3=addr, d_ws2=addr)
    cases = [("qwen3_moe", "d_w3"), ("capacity_top2_bf16", "d_b1"),
             ("capacity_top2_bf16", "d_b2"), ("deepseek_v3_block", "d_ws2")]
    for name, missing in cases:
        cfg = M.make_config(W.WORKLOADS[name])
        n = ctypes.c_size_t()
        assert lib.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 0
        fw = ctypes.c_size_t()
        lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(fw))
        assert n.value > fw.value
        ww = M.MoEWeights(w_router=addr, w1=addr, w3=addr, w2=addr, b1=addr, b2=addr,
                          ws1=addr, ws3=addr, ws2=addr, sel_bias=addr)
        gg = M.MoEGrads(**{k: (None if k == missing else v) for k, v in full.items()})
        st = lib.moe_backward(ctypes.byref(cfg), addr, ctypes.byref(ww), addr, 0.0,
                              ctypes.byref(gg), addr, n.value, None)
        assert st == M.MOE_ERR_INVALID_ARG, (name, missing)


def test_wait_check_rejects_bad_arguments(lib):
    buf = ctypes.create_string_buffer(4096)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    f = lib.moe_check_wait_timeout
    assert f(None, 4096, 1_000_000, None) == M.MOE_ERR_INVALID_ARG
    assert f(addr, 128, 1_000_000, None) == M.MOE_ERR_INVALID_ARG       # below 256 bytes
    assert f(addr, 4096, 10, None) == M.MOE_ERR_INVALID_ARG             # limit below 1 us
    assert f(addr, 4096, 5_000_000_000, None) == M.MOE_ERR_INVALID_ARG  # above 1 s


def test_grouping_expert_and_combine_calls_reject_bad_arguments(lib):
    """Every stage entry point checks its pointers, weights and workspace
    before it enqueues anything: the addresses here are host memory and each
    call must return at a check (the toy layer: fp32 SiLU-MLP with biases,
    64 tokens)."""
    cfg = M.make_config(W.WORKLOADS["toy_top2_fp32"])
    c = ctypes.byref(cfg)
    buf = ctypes.create_string_buffer(1 << 20)
    a = (ctypes.addressof(buf) + 255) // 256 * 256
    big = 1 << 40                       # claimed workspace size; never touched
    full = M.MoEWeights(w_router=a, b_router=a, w1=a, b1=a, w2=a, b2=a)
    # grouping: (cfg, idx, x, offsets, row_of_slot, token_of_row, x_perm, stats, ws, bytes, stream)
    disp = lib.moe_dispatch_permute
    assert disp(c, a, a, None, a, a, a, None, a, big, None) == -1          # no offsets
    assert disp(c, a, a, a, a, a, None, None, a, big, None) == -1          # x without x_perm
    assert disp(c, a, a, a, a + 4, a, a, None, a, big, None) == -1         # misaligned row_of_slot
    assert disp(c, None, a, a, a, a, a, None, a, big, None) == -1          # no idx
    assert disp(c, a, a, a, a, a, a, None, a, 16, None) == -3              # short workspace
    assert disp(c, a, a, a, a, a, a, None, None, big, None) == -1          # no workspace
    bad_stats = M.MoEStats(counts=a + 4)
    assert disp(c, a, a, a, a, a, a, ctypes.byref(bad_stats), a, big, None) == -1
    # grouping with a per-expert room: (cfg, idx, x, room, offsets, ...)
    room = lib.moe_dispatch_permute_room
    assert room(c, a, a, None, a, a, a, a, None, a, big, None) == -1       # no room
    assert room(c, a, a, a + 4, a, a, a, a, None, a, big, None) == -1      # misaligned room
    assert room(c, a, a, a, None, a, a, a, None, a, big, None) == -1       # no offsets
    assert room(c, a, a, a, a, a, a, None, None, a, big, None) == -1       # x without x_perm
    assert room(c, a, a, a, a, a, a, a, None, a, 16, None) == -3           # short workspace
    # the grouping check: (cfg, idx, offsets, row_of_slot, token_of_row, ws, bytes, stream)
    chk = lib.moe_check_grouping
    assert chk(c, a, None, a, a, a, big, None) == -1                       # no offsets
    assert chk(c, None, a, a, a, a, big, None) == -1                       # no idx
    assert chk(c, a, a, a + 4, a, a, big, None) == -1                      # misaligned rows
    assert chk(c, a, a, a, a, a, 16, None) == -3                           # short workspace
    assert chk(c, a, a, a, a, None, big, None) == -1                       # no workspace
    noalloc = lib.moe_dispatch_permute_noalloc
    assert noalloc(c, a, a, None, a, a, a, None, None) == -1               # no offsets
    assert noalloc(c, None, a, a, a, a, a, None, None) == -1               # no idx
    assert noalloc(c, a, None, a, a, a, a, None, None) == -1               # x_perm without x
    big_n = _bad(n_tokens=70000)                                           # beyond its fixed scratch
    assert noalloc(ctypes.byref(big_n), a, a, a, a, a, a, None, None) == -2
    # expert GEMMs
    no_b1 = M.MoEWeights(w1=a, w2=a, b2=a)
    assert lib.moe_expert_up(c, a, a, ctypes.byref(no_b1), a, a, big, None) == -1
    assert lib.moe_expert_up(c, a, a, None, a, a, big, None) == -1         # no weights
    assert lib.moe_expert_up(c, a, a, ctypes.byref(full), None, a, big, None) == -1   # no h
    assert lib.moe_expert_up(c, a, a, ctypes.byref(full), a, a, 16, None) == -3
    assert lib.moe_expert_up_gather(c, a, None, a, ctypes.byref(full), a, a, big, None) == -1
    no_b2 = M.MoEWeights(w1=a, b1=a, w2=a)
    assert lib.moe_expert_down(c, a, a, ctypes.byref(no_b2), a, a, big, None) == -1
    assert lib.moe_expert_down(c, a, a, ctypes.byref(full), a + 8, a, big, None) == -1  # misaligned y
    no_w2 = M.MoEWeights(w1=a, b1=a, b2=a)
    assert lib.moe_grouped_ffn(c, a, a, ctypes.byref(no_w2), a, a, a, big, None) == -1
    assert lib.moe_grouped_ffn(c, a, None, ctypes.byref(full), a, a, a, big, None) == -1
    swiglu = _bad(expert=W.EXPERT_SWIGLU, has_bias=False, dtype=W.DTYPE_BF16)
    no_w3 = M.MoEWeights(w1=a, w2=a)
    assert lib.moe_expert_up(ctypes.byref(swiglu), a, a, ctypes.byref(no_w3), a, a, big,
                             None) == -1
    # combine: (cfg, y, row_of_slot, w, shared_out, out, ws, bytes, stream)
    assert lib.moe_combine(c, a, a, None, None, a, a, big, None) == -1     # no weights
    assert lib.moe_combine(c, a, a, a, a + 4, a, a, big, None) == -1       # misaligned shared_out
    assert lib.moe_combine(c, a, a, a, None, a, None, big, None) == -1     # no workspace
    # the host-buffer forward and the error read-back
    assert lib.moe_forward_host(c, None, ctypes.byref(full), a, None, a, big, None) == -1
    assert lib.moe_forward_host(c, a, ctypes.byref(full), a, None, a, 16, None) == -3
    code = ctypes.c_int32(7)
    assert lib.moe_read_device_error(None, ctypes.byref(code), None) == -1
    assert lib.moe_read_device_error(a, None, None) == -1
    assert code.value == 7


def test_workspace_sizes_and_reset_on_the_host(lib):
    cfg = M.make_config(W.WORKLOADS["toy_top2_fp32"])
    ws = M.MoEWorkspace(cfg, device="cpu")
    assert ws.nbytes == M.workspace_size(cfg)
    assert M.MoEWorkspace(cfg, device="cpu", forward=False).nbytes == M.scratch_size(cfg)
    ws.tensor[:8] = 7
    ws.reset()
    assert int(ws.tensor.sum()) == 0
