"""Pins of the oracle's backward pass to things other than itself.

The gradients are checked against central finite differences of the (already
pinned) forward oracle, against closed forms, and the tiled order against the
direct form.  CPU only.
"""

import numpy as np
import pytest

import oracle


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.attention_reference(q, k, v, scale, causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences_of_the_forward(causal):
    # dLoss/dX for Loss = sum(O * dO) is exactly what the backward returns.
    rng = np.random.default_rng(7)
    n, d, scale, eps = 6, 4, 0.7, 1e-6
    q, k, v, do = (rng.standard_normal((1, n, d)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * eps)
        assert np.abs(num - g).max() < 1e-7 * max(1.0, np.abs(g).max()), name


def test_uniform_scores_give_closed_forms():
    # All key rows equal -> every score of a row equal -> P = 1/N: dV_j = mean_i dO_i
    # for every key j, and dQ = scale * sum_j dS_ij k = 0 because the dS row sums to 0.
    rng = np.random.default_rng(3)
    n, d = 9, 5
    q = rng.standard_normal((1, n, d))
    k = np.repeat(rng.standard_normal((1, 1, d)), n, axis=1)
    v, do = rng.standard_normal((1, n, d)), rng.standard_normal((1, n, d))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, False)
    assert np.abs(dq).max() < 1e-14
    assert np.abs(dv - do.mean(axis=1, keepdims=True)).max() < 1e-14


def test_causal_last_key_only_sees_the_last_query():
    # Key N-1 is kept only by query N-1, whose softmax weight on it is P[N-1, N-1].
    rng = np.random.default_rng(5)
    n, d, scale = 7, 3, 0.9
    q, k, v, do = (rng.standard_normal((1, n, d)) for _ in range(4))
    _, _, dv = oracle.attention_backward(q, k, v, do, scale, True)
    s = scale * q[0, -1] @ k[0].T
    p_last = np.exp(s[-1] - s.max()) / np.exp(s - s.max()).sum()
    assert np.abs(dv[0, -1] - p_last * do[0, -1]).max() < 1e-14
    # Key 0 is kept by every query: dV_0 = sum_i P[i, 0] dO_i.
    p = oracle.attention_probs(q, k, scale, True)[0]
    assert np.abs(dv[0, 0] - (p[:, 0:1] * do[0]).sum(axis=0)).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,bq,bk", [(37, 7, 5), (64, 16, 16), (1, 16, 16), (100, 128, 128)])
def test_tiled_backward_equals_direct(causal, n, bq, bk):
    rng = np.random.default_rng(n)
    q, k, v, do = (rng.standard_normal((2, n, 8)) for _ in range(4))
    a = oracle.attention_backward(q, k, v, do, 0.35, causal)
    b = oracle.attention_backward_tiled(q, k, v, do, 0.35, causal, bq=bq, bk=bk)
    for x, y in zip(a, b):
        assert np.abs(x - y).max() < 1e-12
