"""Failure detection on the GPU without a fault: the expert GEMMs' bounded
mbarrier wait is made to run out (barriers nothing completes, a 20 ms limit)
through moe_check_wait_timeout.  The device error word reports the timeout,
the other waiting role leaves on the CTA's abort flag, the kernel returns,
and the same context then runs the layer normally."""
import time

import pytest
import torch

from oracle import moe_oracle as O
from routing_dispatch_expert_05_b300 import build as B
from routing_dispatch_expert_05_b300 import moe as M
from tests.parity_util import Device, assert_output_close, inputs_for, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    M.load_library()
    torch.cuda.init()


def test_bounded_wait_times_out_and_the_context_survives():
    inp = inputs_for("toy_top2_fp32", None)
    D = Device(inp)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    M.moe_check_wait_timeout(D.ws, 20_000_000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert M.moe_read_device_error(D.ws) == M.MOE_ERR_TIMEOUT
    flags = D.ws.tensor[128:136].view(torch.int32).cpu().tolist()
    assert flags == [0, 0]                       # neither wait succeeded
    assert 0.015 <= elapsed < 2.0                # gave up after ~20 ms, not 2 s
    # the same context, a cleared error word: the layer runs and is right
    D.ws.tensor[:256].zero_()
    out = D.empty(inp.shape.n_tokens, inp.shape.d_model)
    M.moe_forward(D.cfg, D.t["x"], D.weights, out, None, D.ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_error(D.ws) == M.MOE_OK
    ref = O.forward(inp.shape, inp.values)
    assert_output_close(to_np(out), ref["out_exact"], inp.shape.dtype, "after timeout")
