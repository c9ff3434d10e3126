"""GPU parity of the e4m3 forward with the split exponential switched on
(attn_set_poly_exp2: one exponential pair in four by the polynomial of
csrc/exp2_poly.h on the FMA pipe), against the oracle at the stated FP8
tolerances; and a check that the switch reaches the kernel.
"""

import numpy as np
import pytest
import torch

from tiled_attention_fa2_gb300 import binding, inputs

from parity import TOL_L, TOL_O, errors, make_case, oracle_full, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture
def poly_on(built_library):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    prev = binding.set_poly_exp2(True)
    try:
        yield
    finally:
        binding.set_poly_exp2(prev)


def _check(case, causal, rows=None):
    o, l = run_gpu(case, causal)
    if rows is None:
        o_ref, l_ref = oracle_full(case, causal)
    else:
        o_ref, l_ref = oracle_rows(case, causal, rows)
        o = np.stack([o[h][rows[h]] for h in range(o.shape[0])])
        l = np.stack([l[h][rows[h]] for h in range(l.shape[0])])
    label = f"poly-exp2 e4m3 B{case.B} H{case.H} N{case.N} causal={int(causal)} scale={case.scale:.3g}"
    eo, el = errors(o, l, o_ref, l_ref, label=label)
    assert eo <= TOL_O["e4m3"], f"O max-abs error {eo:.3e}"
    assert el <= TOL_L["e4m3"], f"L max-abs error {el:.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 300, 1000])
def test_poly_exp2_small(poly_on, N, causal):
    _check(make_case(2, 3, N, 128, "e4m3", seed=N + 7), causal)


@pytest.mark.parametrize("scale", [0.02, 0.3, 1.5])
def test_poly_exp2_non_default_scale(poly_on, scale):
    case = make_case(1, 2, 300, 128, "e4m3", seed=int(scale * 100) + 128)
    case.scale_override = scale
    _check(case, True)


def test_poly_exp2_dit_sampled_rows(poly_on):
    w = inputs.WORKLOADS["dit_e4m3"]
    case = make_case(w["B"], w["H"], w["N"], w["d"], w["dtype"])
    _check(case, False, rows=inputs.sample_rows(case.N, case.B, case.H, count=512))


def test_switch_reaches_the_kernel(built_library):
    """The polynomial rounds differently from the exponential unit, so the two
    settings give different bytes on the same inputs (and each is repeatable)."""
    case = make_case(1, 2, 1000, 128, "e4m3", seed=3)
    dev = [t.cuda() for t in case.stored]
    prev = binding.set_poly_exp2(False)
    try:
        o0, l0 = binding.attn_fwd_fp8(*dev, *case.descales)
        binding.set_poly_exp2(True)
        o1, l1 = binding.attn_fwd_fp8(*dev, *case.descales)
        o2, l2 = binding.attn_fwd_fp8(*dev, *case.descales)
    finally:
        binding.set_poly_exp2(prev)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert not torch.equal(l0, l1)
