"""Split-KV forward on the GPU: every split count (automatic included), ragged
N, bf16 d in {64, 128} and e4m3, against the float64 oracle and against the
unsplit path."""

import numpy as np
import pytest
import torch

from tiled_attention_fa2_gb300 import binding

from parity import TOL_L, TOL_O, errors, make_case, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()


def _split_run(case, n_splits):
    dev = [t.cuda() for t in case.stored]
    ds = case.descales if case.dtype == "e4m3" else None
    o, lse = binding.attn_fwd_split(*dev, n_splits=n_splits, descales=ds, scale=case.scale)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
    BH = case.B * case.H
    return (o.double().cpu().numpy().reshape(BH, case.N, case.d),
            lse.double().cpu().numpy().reshape(BH, case.N))


@pytest.mark.parametrize("n_splits", [0, 1, 2, 3, 7])
@pytest.mark.parametrize("N", [100, 300, 1000, 2500])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("e4m3", 128)])
def test_split_matches_oracle(dtype, d, N, n_splits):
    case = make_case(1, 2, N, d, dtype, seed=N + n_splits)
    o, l = _split_run(case, n_splits)
    o_ref, l_ref = oracle_full(case, False)
    eo, el = errors(o, l, o_ref, l_ref, label=f"split{n_splits} {dtype} B1 H2 N{N} d{d} full")
    assert eo <= TOL_O[dtype] and el <= TOL_L[dtype], (eo, el)


def test_split_agrees_with_unsplit_path():
    case = make_case(1, 1, 4096, 128, "bf16", seed=11)
    dev = [t.cuda() for t in case.stored]
    o1, l1 = binding.attn_fwd(*dev)
    o2, l2 = binding.attn_fwd_split(*dev, n_splits=8)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
    assert float((l1 - l2).abs().max()) <= 1e-4


def test_automatic_split_fills_the_device():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s, nbytes = binding.split_plan(1, 2, 8192, 128, 0)
    items = 1 * 2 * (8192 // 256)
    assert s * items >= min(sms, items * 64) or s == 8192 // 128
    assert nbytes > 0
