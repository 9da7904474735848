"""The input generator's bf16 rounding against torch's own fp32 -> bf16
conversion (round to nearest even), on random values, exact ties, values
next to ties, signed zeros, subnormals and infinities; and its token
sub-views."""
import numpy as np
import pytest
import torch

from routing_dispatch_expert_05_b300 import workloads as W


def test_bf16_bits_match_torch_rounding():
    rng = np.random.default_rng(0)
    a = rng.standard_normal(100000).astype(np.float32) * np.float32(3.0)
    u = a.view(np.uint32)
    ties = ((u & 0xFFFF0000) | 0x8000).view(np.float32)          # exactly halfway
    near = ((u & 0xFFFF0000) | 0x7FFF).view(np.float32)          # just below halfway
    special = np.array([0.0, -0.0, 1e-40, -1e-40, np.inf, -np.inf, 3.4e38, -3.4e38],
                       np.float32)
    for arr in (a, ties, near, special):
        want = torch.from_numpy(arr).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(W.bf16_bits(arr).view(np.int16), want)


def test_first_tokens_views_and_refuses_more_tokens_than_it_holds():
    """A sub-view keeps the layer's parameters and shortens x (values and bf16
    bits) to its n tokens; asking for more tokens than the inputs hold is an
    error, since the config would then declare rows that x does not have."""
    inp = W.make_inputs(W.WORKLOADS["capacity_top2_bf16"])
    n_all = inp.shape.n_tokens
    sub = inp.first_tokens(100)
    assert sub.shape.n_tokens == 100
    assert sub.values["x"].shape == (100, inp.shape.d_model)
    assert sub.bits["x"].shape == (100, inp.shape.d_model)
    assert sub.values["w1"] is inp.values["w1"]
    assert inp.first_tokens(0).values["x"].shape[0] == 0
    assert inp.first_tokens(n_all).values["x"].shape[0] == n_all
    with pytest.raises(ValueError):
        inp.first_tokens(n_all + 1)
    with pytest.raises(ValueError):
        inp.first_tokens(-1)
