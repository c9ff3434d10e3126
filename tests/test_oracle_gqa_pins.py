"""Pins of the oracle's grouped-query attention (CPU, float64).

Grouped-query attention ("Kernels and Memory in LLM Inference", "Store less:
MQA, GQA, MLA", "Grouped-query attention (2023)") splits the query heads into
groups that each read one K/V head; one group is multi-query attention and one
group per head is ordinary multi-head attention.  What pins the oracle's head
map and its use:

* the two ends of the dial the page names: H_kv = H is multi-head attention
  (the already pinned definition, head by head) and H_kv = 1 is multi-query
  attention (every query head against the single K/V head);
* materialising the sharing: repeating each K/V head for the query heads of
  its group gives an ordinary multi-head problem with the same O and L;
* an independent implementation: PyTorch's float64 CPU
  scaled_dot_product_attention with enable_gqa=True;
* a planted mistake (heads grouped round-robin, h mod H_kv, instead of in
  consecutive runs) disagrees with that implementation.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _inputs(B, H, hkv, n, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, n, d), dtype=torch.float64, generator=g)
    k = torch.randn((B, hkv, n, d), dtype=torch.float64, generator=g)
    v = torch.randn((B, hkv, n, d), dtype=torch.float64, generator=g)
    return q, k, v


def test_head_map_groups_consecutive_heads():
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 8, 8) for h in range(8)] == list(range(8))
    assert [oracle.kv_head_of(h, 8, 1) for h in range(8)] == [0] * 8
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 8, 3)


@pytest.mark.parametrize("causal", [False, True])
def test_one_kv_head_per_query_head_is_multi_head(causal):
    q, k, v = _inputs(2, 4, 4, 45, 16, seed=1)
    o, lse = oracle.attention_gqa(q.numpy(), k.numpy(), v.numpy(), 0.3, causal)
    o_ref, l_ref = oracle.attention_reference(q.numpy(), k.numpy(), v.numpy(), 0.3, causal)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, l_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_one_kv_head_is_multi_query(causal):
    q, k, v = _inputs(2, 3, 1, 37, 8, seed=2)
    o, lse = oracle.attention_gqa(q.numpy(), k.numpy(), v.numpy(), 0.5, causal)
    for b in range(2):
        for h in range(3):
            o_ref, l_ref = oracle.attention_reference(q[b, h].numpy(), k[b, 0].numpy(), v[b, 0].numpy(), 0.5,
                                                      causal)
            assert np.array_equal(o[b, h], o_ref) and np.array_equal(lse[b, h], l_ref)


@pytest.mark.parametrize("H,hkv", [(8, 2), (6, 3), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_repeated_kv_heads_give_the_same_result(H, hkv, causal):
    q, k, v = _inputs(2, H, hkv, 50, 16, seed=H + hkv)
    rep = H // hkv
    k_full = np.repeat(k.numpy(), rep, axis=1)
    v_full = np.repeat(v.numpy(), rep, axis=1)
    o, lse = oracle.attention_gqa(q.numpy(), k.numpy(), v.numpy(), 0.25, causal)
    o_ref, l_ref = oracle.attention_reference(q.numpy(), k_full, v_full, 0.25, causal)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, l_ref)


@pytest.mark.parametrize("H,hkv", [(8, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_enable_gqa(H, hkv, causal):
    q, k, v = _inputs(1, H, hkv, 70, 32, seed=10 * H + hkv)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.2, enable_gqa=True).numpy()
    o, _ = oracle.attention_gqa(q.numpy(), k.numpy(), v.numpy(), 0.2, causal)
    assert np.abs(o - ref).max() < 1e-12


def test_rows_match_the_full_result():
    q, k, v = _inputs(2, 4, 2, 90, 16, seed=7)
    rng = np.random.default_rng(3)
    rows = np.stack([np.sort(rng.choice(90, 12, replace=False)) for _ in range(8)])
    o, lse = oracle.attention_gqa(q.numpy(), k.numpy(), v.numpy(), 0.4, True)
    o_r, l_r = oracle.attention_gqa_rows(q.numpy(), k.numpy(), v.numpy(), rows, 0.4, True)
    for bh in range(8):
        b, h = divmod(bh, 4)
        assert np.array_equal(o_r[bh], o[b, h][rows[bh]])
        assert np.array_equal(l_r[bh], lse[b, h][rows[bh]])


def test_planted_round_robin_grouping_is_caught():
    H, hkv = 8, 2
    q, k, v = _inputs(1, H, hkv, 40, 16, seed=5)
    ref = F.scaled_dot_product_attention(q, k, v, scale=0.2, enable_gqa=True).numpy()
    wrong = np.empty_like(ref)
    for h in range(H):
        g = h % hkv  # the mistake: round-robin instead of consecutive groups
        wrong[0, h], _ = oracle.attention_reference(q[0, h].numpy(), k[0, g].numpy(), v[0, g].numpy(), 0.2)
    assert np.abs(wrong - ref).max() > 1e-2
