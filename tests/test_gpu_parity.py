"""GPU vs float64 oracle, element by element, on seeded inputs.

Small shapes (many tiles, ragged tails, N=1, both head dims, causal and not)
are compared in full; the five named workloads are compared in full where the
oracle is tractable and on 512 seeded rows per head (rows 0 and N-1 included)
on the two largest, in the same launch configuration the bench times.
"""

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_fa2_gb300 import binding, inputs

from parity import TOL_F32_TIGHT, TOL_L, TOL_O, errors, make_case, oracle_full, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(built_library):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()


def _check(case, causal, rows=None, tight=None, tol_o=None):
    o, l = run_gpu(case, causal)
    if rows is None:
        o_ref, l_ref = oracle_full(case, causal)
    else:
        o_ref, l_ref = oracle_rows(case, causal, rows)
        o = np.stack([o[h][rows[h]] for h in range(o.shape[0])])
        l = np.stack([l[h][rows[h]] for h in range(l.shape[0])])
    label = getattr(case, "name", "") + f" {case.dtype} B{case.B} H{case.H} N{case.N} d{case.d} causal={int(causal)} " + (
        "full" if rows is None else f"{rows.shape[1]} rows/head")
    eo, el = errors(o, l, o_ref, l_ref, label=label)
    assert eo <= (TOL_O[case.dtype] if tol_o is None else tol_o), f"O max-abs error {eo:.3e}"
    assert el <= TOL_L[case.dtype], f"L max-abs error {el:.3e}"
    if tight is not None:
        assert eo <= tight and el <= tight, f"tight check: O {eo:.3e} L {el:.3e}"
    return eo, el


# ------------------------------------------------------------ small shapes, full compare

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 37, 100, 128, 200, 300])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_f32_small(N, d, causal):
    _check(make_case(2, 3, N, d, "f32", seed=N + d), causal, tight=TOL_F32_TIGHT)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 37, 100, 127, 128, 129, 255, 256, 257, 300, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_small(N, d, causal):
    _check(make_case(2, 3, N, d, "bf16", seed=N + d), causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 256, 300, 1000])
def test_e4m3_small(N, causal):
    _check(make_case(2, 3, N, 128, "e4m3", seed=N), causal)


@pytest.mark.parametrize("q_mult", [8.0, 32.0])
def test_bf16_max_moves_between_tiles(q_mult):
    """Large score range: the running max changes across key tiles, so the
    alpha rescale of O is exercised (and checked) many times."""
    _check(make_case(1, 4, 1000, 128, "bf16", seed=5, q_mult=q_mult), False)
    _check(make_case(1, 4, 1000, 64, "bf16", seed=6, q_mult=q_mult), True)


def test_many_heads_small_n():
    _check(make_case(8, 64, 64, 64, "bf16", seed=9), True)


# ------------------------------------------------------------ named workloads

def _wl(name):
    w = inputs.WORKLOADS[name]
    case = make_case(w["B"], w["H"], w["N"], w["d"], w["dtype"], q_mult=w["q_mult"])
    case.name = name
    return case, w["causal"]


def test_tiny_f32_workload():
    case, causal = _wl("tiny_f32")
    _check(case, causal, tight=TOL_F32_TIGHT)


@pytest.mark.parametrize("name", ["prefill_causal_bf16", "sweep_d64_bf16", "sweep_d128_bf16",
                                  "sweep_d64_bf16_qx8", "sweep_d128_bf16_qx8"])
def test_full_compare_workloads(name):
    case, causal = _wl(name)
    _check(case, causal)


@pytest.mark.parametrize("name", ["dit_e4m3", "long_causal_bf16", "long_causal_e4m3"])
def test_sampled_rows_workloads(name):
    case, causal = _wl(name)
    rows = inputs.sample_rows(case.N, case.B, case.H, count=512)
    _check(case, causal, rows=rows)


# ------------------------------------------------------------ properties

def test_repeat_is_bit_exact():
    case = make_case(2, 4, 777, 128, "bf16", seed=1)
    dev = [t.cuda() for t in case.stored]
    o1, l1 = binding.attn_fwd(*dev, causal=True)
    o2, l2 = binding.attn_fwd(*dev, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "e4m3"])
def test_host_entry_matches_device_entry(dtype):
    case = make_case(1, 2, 300, 128 if dtype != "f32" else 64, dtype, seed=2)
    dev = [t.cuda() for t in case.stored]
    if dtype == "e4m3":
        o_d, l_d = binding.attn_fwd_fp8(*dev, *case.descales, causal=True)
    else:
        o_d, l_d = binding.attn_fwd(*dev, causal=True)
    h = [t.pin_memory() for t in case.stored]
    h_o = torch.empty(o_d.shape, dtype=o_d.dtype).pin_memory()
    h_l = torch.empty(l_d.shape, dtype=torch.float32).pin_memory()
    d_in = [torch.empty_like(t) for t in dev]
    d_o, d_l = torch.empty_like(o_d), torch.empty_like(l_d)
    binding.attn_fwd_host(*h, h_o, h_l, *d_in, d_o, d_l, causal=True, descales=case.descales)
    torch.cuda.synchronize()
    assert torch.equal(h_o, o_d.cpu()) and torch.equal(h_l, l_d.cpu())


def test_outputs_outside_the_valid_rows_are_untouched():
    """Rows past N are never written: a guard band after O and L keeps its sentinel."""
    case = make_case(1, 1, 300, 128, "bf16", seed=4)
    q, k, v = [t.cuda() for t in case.stored]
    o_big = torch.full((1, 1, 300 + 64, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    l_big = torch.full((1, 1, 300 + 64), 7.0, dtype=torch.float32, device="cuda")
    o = o_big[:, :, :300]
    l = l_big[:, :, :300]
    lib = binding.load_library()
    st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), 1, 1, 300, 128,
                      case.scale, 0, 1, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert bool((o_big[:, :, 300:] == 7.0).all()) and bool((l_big[:, :, 300:] == 7.0).all())


def test_device_status_is_clean():
    assert binding.get_device_status() == 0


# ------------------------------------------------------------ softmax scale other than 1/sqrt(d)

@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("e4m3", 128), ("f32", 64)])
@pytest.mark.parametrize("scale", [0.02, 0.3, 1.5])
@pytest.mark.parametrize("causal", [False, True])
def test_non_default_scale(dtype, d, scale, causal):
    """The scale multiplies the scores before the softmax (1.5 on unit-variance
    inputs spreads a row over about 30 doublings, so the reference max moves).

    e4m3: a large scale makes rows peaked.  P goes through e4m3 (3 mantissa
    bits), and the kernel divides O by the sum of exactly those rounded weights,
    so a row's dominant weight carries no rounding error into O and the stated
    6e-2 bar holds here too; L comes from the unrounded sum (1e-3)."""
    case = make_case(1, 2, 300, d, dtype, seed=int(scale * 100) + d)
    case.scale_override = scale
    _check(case, causal, tight=TOL_F32_TIGHT if dtype == "f32" else None)
