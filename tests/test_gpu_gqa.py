"""GPU parity of grouped-query attention (attn_fwd_gqa) against the oracle.

Query heads are split into groups that read one K/V head each ("Kernels and
Memory in LLM Inference", "Store less: MQA, GQA, MLA", "Grouped-query
attention (2023)"); the oracle's head map (``oracle.kv_head_of``) picks the
K/V head, and each query head is compared with the oracle's definition.
Group sizes H / H_kv in {1, 4, 8} (8 with H_kv = 1 is multi-query attention),
every tensor-core dtype and head dimension, causal and not, ragged N.
"""

import numpy as np
import pytest
import torch

from tiled_attention_fa2_gb300 import binding, inputs

from parity import TOL_F32_TIGHT, TOL_L, TOL_O, errors, make_case, oracle_full, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu


def _check(case, causal, rows=None, tight=None):
    o, l = run_gpu(case, causal)
    if rows is None:
        o_ref, l_ref = oracle_full(case, causal)
    else:
        o_ref, l_ref = oracle_rows(case, causal, rows)
        o = np.stack([o[h][rows[h]] for h in range(o.shape[0])])
        l = np.stack([l[h][rows[h]] for h in range(l.shape[0])])
    label = f"gqa {case.dtype} B{case.B} H{case.H} Hkv{case.Hkv or case.H} N{case.N} d{case.d} causal={int(causal)}"
    eo, el = errors(o, l, o_ref, l_ref, label=label)
    assert eo <= TOL_O[case.dtype], f"O max-abs error {eo:.3e}"
    assert el <= TOL_L[case.dtype], f"L max-abs error {el:.3e}"
    if tight is not None:
        assert eo <= tight and el <= tight, f"tight check: O {eo:.3e} L {el:.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [8, 2, 1])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("e4m3", 128)])
def test_gqa_small(dtype, d, hkv, causal):
    case = make_case(2, 8, 300, d, dtype, seed=hkv + d, n_kv_heads=hkv)
    _check(case, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hkv", [4, 1])
def test_gqa_f32(hkv, causal):
    case = make_case(1, 4, 200, 64, "f32", seed=3, n_kv_heads=hkv)
    _check(case, causal, tight=TOL_F32_TIGHT)


@pytest.mark.parametrize("N", [1, 129, 1000])
def test_gqa_ragged_lengths(N):
    _check(make_case(1, 16, N, 128, "bf16", seed=N, n_kv_heads=2), True)


def test_gqa_with_one_group_per_head_equals_multi_head():
    """H_kv = H through attn_fwd_gqa gives exactly attn_fwd's bytes."""
    case = make_case(2, 4, 500, 128, "bf16", seed=4)
    dev = [t.cuda() for t in case.stored]
    o1, l1 = binding.attn_fwd(*dev, causal=True)
    o2, l2 = binding.attn_fwd_gqa(*dev, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_equals_multi_head_on_repeated_kv_heads():
    """Materialising the sharing (each K/V head repeated for its group) and
    running the multi-head kernel gives the same bytes."""
    case = make_case(1, 8, 700, 128, "e4m3", seed=5, n_kv_heads=2)
    q, k, v = (t.cuda() for t in case.stored)
    o1, l1 = binding.attn_fwd_gqa(q, k, v, descales=case.descales, causal=False)
    kr, vr = (t.repeat_interleave(4, dim=1).contiguous() for t in (k, v))
    o2, l2 = binding.attn_fwd_fp8(q, kr, vr, *case.descales, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["prefill_gqa_bf16", "prefill_gqa_e4m3"])
def test_gqa_workloads_sampled_rows(name):
    w = inputs.WORKLOADS[name]
    case = make_case(w["B"], w["H"], w["N"], w["d"], w["dtype"], q_mult=w["q_mult"], n_kv_heads=w["Hkv"])
    rows = inputs.sample_rows(case.N, case.B, case.H, count=512)
    _check(case, w["causal"], rows=rows)


def test_gqa_rejects_heads_not_divisible():
    case = make_case(1, 6, 128, 128, "bf16", seed=6, n_kv_heads=4)
    dev = [t.cuda() for t in case.stored]
    with pytest.raises(binding.AttnError) as e:
        binding.attn_fwd_gqa(*dev)
    assert e.value.status == 1
