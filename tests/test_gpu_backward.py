"""GPU parity of the backward pass against the float64 oracle.

The CUDA forward produces O and L, the CUDA backward the gradients; the oracle
computes the gradients from the same bf16 Q, K, V and dO bytes in float64.
Tolerance: max |GPU - oracle| <= 2e-2 * max |oracle| + 2e-3 per gradient (P and
dS enter the tensor-core products rounded to bf16, relative 2^-9, and each
gradient is stored as bf16, relative 2^-9; D = rowsum(dO * O) uses the bf16 O).
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_fa2_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CASES = [(1, 2, n, d, c) for n in (1, 37, 128, 200, 300) for d in (64, 128) for c in (False, True)]
CASES += [(2, 3, 513, 128, True), (1, 1, 1000, 64, False)]


def run_case(B, H, N, d, causal, seed):
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=seed)
    do = inputs.make_dout_f32(B, H, N, d, seed=seed + 1)
    qb, kb, vb, dob = (inputs.to_bf16(t) for t in (q, k, v, do))
    dev = [t.cuda() for t in (qb, kb, vb, dob)]
    o, lse = binding.attn_fwd(dev[0], dev[1], dev[2], causal=causal)
    dq, dk, dv = binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], causal=causal)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    ref = oracle.attention_backward(*(t.double().numpy() for t in (qb, kb, vb, dob)), 1.0 / np.sqrt(d), causal)
    return [g.float().cpu().double().numpy() for g in (dq, dk, dv)], ref


@pytest.mark.parametrize("B,H,N,d,causal", CASES)
def test_backward_matches_oracle(B, H, N, d, causal):
    got, ref = run_case(B, H, N, d, causal, seed=N + d)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), name
        err = np.abs(g - r).max()
        tol = 2e-2 * np.abs(r).max() + 2e-3
        assert err <= tol, f"{name}: max abs error {err:.3e} > {tol:.3e} (max |ref| {np.abs(r).max():.3e})"


def test_backward_is_deterministic_except_for_dq_rounding():
    # dK and dV accumulate in TMEM in a fixed order: bit-identical on a repeat.
    # dQ is a sum of fp32 atomic adds, whose order may vary: equal within 1e-3.
    a, _ = run_case(1, 2, 300, 128, True, seed=5)
    b, _ = run_case(1, 2, 300, 128, True, seed=5)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= 1e-3 * max(1.0, np.abs(a[0]).max())


def test_backward_on_the_causal_prefill_shape_sampled_heads():
    # The full causal prefill shape (B=4, H=16, N=2048, d=128) through the CUDA
    # forward and backward; three heads (first, a middle one, last) compared in full.
    B, H, N, d = 4, 16, 2048, 128
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=11)
    do = inputs.make_dout_f32(B, H, N, d, seed=12)
    qb, kb, vb, dob = (inputs.to_bf16(t) for t in (q, k, v, do))
    dev = [t.cuda() for t in (qb, kb, vb, dob)]
    o, lse = binding.attn_fwd(dev[0], dev[1], dev[2], causal=True)
    grads = binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], causal=True)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    got = [g.float().cpu().reshape(B * H, N, d) for g in grads]
    flat = [t.reshape(B * H, N, d) for t in (qb, kb, vb, dob)]
    for h in (0, 27, B * H - 1):
        ref = oracle.attention_backward(*(t[h].double().numpy() for t in flat), 1.0 / np.sqrt(d), True)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            err = np.abs(g[h].double().numpy() - r).max()
            tol = 2e-2 * np.abs(r).max() + 2e-3
            assert err <= tol, f"head {h} {name}: {err:.3e} > {tol:.3e}"


@pytest.mark.parametrize("scale", [0.02, 0.5])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_non_default_scale(scale, causal):
    B, H, N, d = 1, 2, 300, 128
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=21)
    do = inputs.make_dout_f32(B, H, N, d, seed=22)
    qb, kb, vb, dob = (inputs.to_bf16(t) for t in (q, k, v, do))
    dev = [t.cuda() for t in (qb, kb, vb, dob)]
    o, lse = binding.attn_fwd(dev[0], dev[1], dev[2], scale=scale, causal=causal)
    grads = binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    ref = oracle.attention_backward(*(t.double().numpy() for t in (qb, kb, vb, dob)), scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        err = np.abs(g.float().cpu().double().numpy() - r).max()
        tol = 2e-2 * np.abs(r).max() + 2e-3
        assert err <= tol, f"{name}: {err:.3e} > {tol:.3e}"


@pytest.mark.parametrize("order", ["key", "head"])
@pytest.mark.parametrize("d", [64, 128])
def test_causal_backward_in_either_grid_order(order, d, monkeypatch):
    # A causal backward deals its items key-tile-major (the default) or
    # head-major (ATTN_BWD_GRID_ORDER=head).  Both match the oracle.
    monkeypatch.setenv("ATTN_BWD_GRID_ORDER", order)
    got, ref = run_case(2, 3, 513, d, True, seed=31 + d)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        err = np.abs(g - r).max()
        tol = 2e-2 * np.abs(r).max() + 2e-3
        assert err <= tol, f"{order} {name}: {err:.3e} > {tol:.3e}"


def _grads(B, H, N, d, causal, seed):
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=seed)
    do = inputs.make_dout_f32(B, H, N, d, seed=seed + 1)
    dev = [inputs.to_bf16(t).cuda() for t in (q, k, v, do)]
    o, lse = binding.attn_fwd(dev[0], dev[1], dev[2], causal=causal)
    grads = binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], causal=causal)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    return [g.float().cpu() for g in grads]


def test_long_causal_backward_is_the_same_in_both_grid_orders(monkeypatch):
    # The long causal shape (B=1, H=8, N=32768, d=128): each work item computes
    # the dK, dV rows of its own key tile whatever the order, so they are
    # bit-identical across the orders; dQ differs only by the order of its fp32
    # reduce-adds.
    monkeypatch.setenv("ATTN_BWD_GRID_ORDER", "head")
    a = _grads(1, 8, 32768, 128, True, seed=41)
    monkeypatch.delenv("ATTN_BWD_GRID_ORDER")
    b = _grads(1, 8, 32768, 128, True, seed=41)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert float((a[0] - b[0]).abs().max()) <= 1e-3 * max(1.0, float(a[0].abs().max()))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_outputs_outside_the_valid_rows_are_untouched(d, causal):
    """Rows past N of dq, dk and dv are never written (at d = 128 dV and dK leave
    through TMA stores that the tensor map clips at N): a guard band after each
    output keeps its sentinel, and dK, dV equal those of a call without it."""
    N = 300
    q, k, v = inputs.make_qkv_f32(1, 1, N, d, seed=9)
    do = inputs.make_dout_f32(1, 1, N, d, seed=10)
    dev = [inputs.to_bf16(t).cuda() for t in (q, k, v, do)]
    o, lse = binding.attn_fwd(dev[0], dev[1], dev[2], causal=causal)
    bigs = [torch.full((1, 1, N + 64, d), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    outs = [b[:, :, :N] for b in bigs]
    binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], dq=outs[0], dk=outs[1], dv=outs[2], causal=causal)
    ref = binding.attn_bwd(dev[0], dev[1], dev[2], o, lse, dev[3], causal=causal)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    for name, big in zip(("dq", "dk", "dv"), bigs):
        assert bool((big[:, :, N:] == 7.0).all()), name
    assert torch.equal(outs[1], ref[1]) and torch.equal(outs[2], ref[2])
