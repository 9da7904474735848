"""The input generator's bf16 rounding against torch's own fp32 -> bf16
conversion (round to nearest even), on random values, exact ties, values
next to ties, signed zeros, subnormals and infinities."""
import numpy as np
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
