"""The seeded input recipe and the workload accounting (no GPU).

The same generator feeds the GPU tests, the bench and the oracle's callers, so
its properties are checked here: determinism, the order Q, K, V, the exact
power-of-two multiplier, the FP8 absmax scale, the sampled rows, and the
algorithmic FLOP count of each named workload (4 B H N^2 d, halved for causal,
the counting of the bench harness in "FlashAttention-2 from PyTorch to Triton").
"""

import numpy as np
import pytest
import torch

from tiled_attention_fa2_gb300 import inputs


def test_generator_is_deterministic_and_draws_q_then_k_then_v():
    q1, k1, v1 = inputs.make_qkv_f32(1, 2, 33, 16, seed=7)
    q2, k2, v2 = inputs.make_qkv_f32(1, 2, 33, 16, seed=7)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    g = torch.Generator(device="cpu").manual_seed(7)
    draws = [torch.randn((1, 2, 33, 16), dtype=torch.float32, generator=g) for _ in range(3)]
    assert torch.equal(q1, draws[0]) and torch.equal(k1, draws[1]) and torch.equal(v1, draws[2])
    q3, _, _ = inputs.make_qkv_f32(1, 2, 33, 16, seed=8)
    assert not torch.equal(q1, q3)


def test_q_multiplier_is_exact():
    q1, k1, _ = inputs.make_qkv_f32(1, 1, 50, 8, seed=3)
    q8, k8, _ = inputs.make_qkv_f32(1, 1, 50, 8, seed=3, q_mult=8.0)
    assert torch.equal(q8, q1 * 8.0) and torch.equal(k8, k1)
    assert torch.equal(inputs.to_bf16(q8).float(), inputs.to_bf16(q1).float() * 8.0)


def test_e4m3_absmax_maps_to_the_largest_code():
    x, _, _ = inputs.make_qkv_f32(1, 1, 64, 32, seed=5)
    codes, descale = inputs.quantize_e4m3(x)
    amax = float(x.abs().max())
    assert descale == pytest.approx(amax / 448.0, rel=1e-6)
    flat = x.flatten()
    i = int(flat.abs().argmax())
    # 0x7E is +448 in E4M3 (exponent 1111, mantissa 110), 0xFE is -448
    assert int(codes.flatten()[i]) == (0x7E if float(flat[i]) > 0 else 0xFE)
    assert codes.dtype == torch.uint8 and codes.shape == x.shape


@pytest.mark.parametrize("N,count", [(30272, 512), (32768, 512), (700, 64)])
def test_sampled_rows_hold_first_and_last_and_are_distinct(N, count):
    rows = inputs.sample_rows(N, 1, 3, count=count)
    assert rows.shape == (3, count)
    for r in rows:
        assert r[0] == 0 and r[-1] == N - 1
        assert np.all(np.diff(r) > 0)  # sorted, distinct
    assert not np.array_equal(rows[0], rows[1])  # one seed per head
    assert np.array_equal(rows, inputs.sample_rows(N, 1, 3, count=count))


def test_sampled_rows_are_all_rows_for_short_heads():
    rows = inputs.sample_rows(300, 2, 2, count=512)
    assert rows.shape == (4, 300)
    assert all(np.array_equal(r, np.arange(300)) for r in rows)


# Algorithmic FLOPs per call of the workloads (4 B H N^2 d, halved for causal).
@pytest.mark.parametrize("name,flops", [
    ("tiny_f32", 33.554432e6),
    ("prefill_causal_bf16", 68.719476736e9),
    ("sweep_d64_bf16", 274.877906944e9),
    ("sweep_d128_bf16", 549.755813888e9),
    ("dit_e4m3", 26.274848309248e12),
    ("long_causal_bf16", 2.199023255552e12),
])
def test_workload_flops(name, flops):
    w = inputs.WORKLOADS[name]
    got = inputs.attention_flops(w["B"], w["H"], w["N"], w["d"], w["causal"])
    assert got == pytest.approx(flops, rel=1e-4)
