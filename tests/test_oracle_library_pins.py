"""Pins of the oracle to an independent library implementation (CPU, float64).

PyTorch's scaled_dot_product_attention on the CPU in float64 computes the same
definition (scores scaled, causal keys j <= i, row softmax, weighted sum of V),
and autograd through it applies the chain rule with code of its own.  The
oracle's forward and backward must agree with both to float64 rounding, on
sizes and scales the brute-force and finite-difference pins do not reach.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _inputs(n, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((2, n, d), dtype=torch.float64, generator=g) for _ in range(4)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d,scale", [(200, 64, 0.125), (129, 128, 0.088), (33, 16, 1.3)])
def test_forward_matches_torch_sdpa(n, d, scale, causal):
    q, k, v, _ = _inputs(n, d, seed=n + d)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale).numpy()
    o, _ = oracle.attention_reference(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    assert np.abs(o - ref).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d,scale", [(70, 16, 0.25), (128, 64, 0.125), (17, 8, 1.1)])
def test_backward_matches_torch_autograd(n, d, scale, causal):
    q, k, v, do = _inputs(n, d, seed=3 * n + d)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = F.scaled_dot_product_attention(qa, ka, va, is_causal=causal, scale=scale)
    (out * do).sum().backward()
    dq, dk, dv = oracle.attention_backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), scale, causal)
    for name, mine, ref in (("dq", dq, qa.grad), ("dk", dk, ka.grad), ("dv", dv, va.grad)):
        ref = ref.numpy()
        assert np.abs(mine - ref).max() < 1e-11 * max(1.0, np.abs(ref).max()), name
