"""Pins for the float64 oracle: it is checked against things other than itself.

* values printed on the pages (tests/golden/, with citations);
* closed forms (identical keys, a dominant key, the causal first row);
* invariants (rows of P sum to 1, key permutation, per-row score shift, scale
  folding);
* a 40-digit brute force written with plain loops (mpmath), on tiny inputs;
* a library routine the oracle does not use (scipy.special.logsumexp);
* the tile-by-tile online-softmax re-derivation against the definition;
* the e4m3 / bf16 decoders against the format definition and against torch.

The mutation tests at the end plant plausible mistakes in the oracle (on the
CPU) and check that the brute-force pin catches each of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oracle_attention
from tiled_attention_fa2_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- worked example


def _worked_example(golden):
    g = golden("online_softmax_worked_example.txt")
    scores = np.array(g["scores"][0])
    q = np.ones((1, 1))
    k = scores.reshape(4, 1)
    v = np.eye(4)
    return g, q, k, v


def test_worked_example_final_weights(golden):
    """Online softmax example of the FP8 RTX 5080 page: O row = printed weights."""
    g, q, k, v = _worked_example(golden)
    o, lse = oracle.attention_reference(q, k, v, scale=1.0)
    w, tol = g["weights"]
    np.testing.assert_allclose(o[0], w, atol=tol)
    lv, ltol = g["l"]
    m = g["strip1_m"][0][0]
    assert abs(math.exp(lse[0] - m) - lv[0]) <= ltol
    un, utol = g["unnormalised"]
    np.testing.assert_allclose(o[0] * math.exp(lse[0] - m), un, atol=utol)


def test_worked_example_strip_states(golden):
    """Strip 0 alone gives m=2, l=1.368; the second strip's alpha is 0.135."""
    g, q, k, v = _worked_example(golden)
    _, lse0 = oracle.attention_tiled(q, k[:2], v[:2], scale=1.0, bq=1, bk=2)
    m0 = g["strip0_m"][0][0]
    l0, tol = g["strip0_l"]
    assert abs(math.exp(lse0[0] - m0) - l0[0]) <= tol
    a, atol = g["strip1_alpha"]
    assert abs(math.exp(m0 - g["strip1_m"][0][0]) - a[0]) <= atol
    # two strips of two keys reproduce the whole-row result
    o_t, l_t = oracle.attention_tiled(q, k, v, scale=1.0, bq=1, bk=2)
    o_n, l_n = oracle.attention_reference(q, k, v, scale=1.0)
    np.testing.assert_allclose(o_t, o_n, atol=1e-15)
    np.testing.assert_allclose(l_t, l_n, atol=1e-15)


# ---------------------------------------------------------------- brute force


def _mp_attention(q, k, v, scale, causal):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    n, d = q.shape
    nk = k.shape[0]
    o = np.empty((n, v.shape[1]))
    lse = np.empty(n)
    for i in range(n):
        s = []
        for j in range(nk):
            if causal and j > i:
                continue
            acc = mpmath.mpf(0)
            for c in range(d):
                acc += mpmath.mpf(float(q[i, c])) * mpmath.mpf(float(k[j, c]))
            s.append((j, acc * mpmath.mpf(scale)))
        z = mpmath.fsum(mpmath.exp(x) for _, x in s)
        lse[i] = float(mpmath.log(z))
        for c in range(v.shape[1]):
            o[i, c] = float(mpmath.fsum(mpmath.exp(x) * mpmath.mpf(float(v[j, c])) for j, x in s) / z)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 3), (5, 4), (9, 2)])
def test_matches_high_precision_brute_force(n, d, causal):
    rng = np.random.default_rng(7 + n + d)
    q, k, v = (rng.standard_normal((n, d)) * 2 for _ in range(3))
    scale = 1 / math.sqrt(d)
    o_ref, l_ref = _mp_attention(q, k, v, scale, causal)
    o, lse = oracle.attention_reference(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, l_ref, rtol=0, atol=1e-13)
    o_t, l_t = oracle.attention_tiled(q, k, v, scale, causal, bq=2, bk=3)
    np.testing.assert_allclose(o_t, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_t, l_ref, rtol=0, atol=1e-13)


def test_lse_matches_scipy_logsumexp():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((2, 3, 37, 16)) for _ in range(3))
    scale = 0.25
    _, lse = oracle.attention_reference(q, k, v, scale)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    np.testing.assert_allclose(lse, special.logsumexp(s, axis=-1), rtol=0, atol=1e-12)
    # causal: masked scores are excluded (-inf), as the FA2 tutorial's test does
    _, lse_c = oracle.attention_reference(q, k, v, scale, causal=True)
    s_c = np.where(np.tril(np.ones((37, 37), bool)), s, -np.inf)
    np.testing.assert_allclose(lse_c, special.logsumexp(s_c, axis=-1), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms


def test_probability_rows_sum_to_one():
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((2, 50, 8)) * 3, rng.standard_normal((2, 50, 8)) * 3
    for causal in (False, True):
        p = oracle.attention_probs(q, k, 0.5, causal)
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p[0], 1) == 0)


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(5)
    n, d = 33, 8
    q = rng.standard_normal((n, d))
    k = np.tile(rng.standard_normal((1, d)), (n, 1))
    v = rng.standard_normal((n, d))
    scale = 0.3
    o, lse = oracle.attention_reference(q, k, v, scale)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (n, 1)), rtol=0, atol=1e-13)
    s = scale * (q @ k[0])
    np.testing.assert_allclose(lse, s + math.log(n), rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value_row():
    n, d = 40, 4
    rng = np.random.default_rng(9)
    k = rng.standard_normal((n, d)) * 0.01
    q = np.zeros((n, d))
    q[:, 0] = 1.0
    j_star = 17
    k[j_star, 0] = 60.0  # score 60 above the others (which are ~0)
    v = rng.standard_normal((n, d))
    o, lse = oracle.attention_reference(q, k, v, 1.0)
    bound = n * math.exp(-59.0) * np.abs(v).max() * 2
    np.testing.assert_allclose(o, np.tile(v[j_star], (n, 1)), rtol=0, atol=bound)
    np.testing.assert_allclose(lse, k[j_star, 0] + np.log1p((n - 1) * np.exp(-60.0)), atol=1e-9)


def test_causal_first_row_is_v0_and_last_row_is_full():
    rng = np.random.default_rng(2)
    q, k, v = (rng.standard_normal((3, 21, 6)) for _ in range(3))
    scale = 0.7
    o, lse = oracle.attention_reference(q, k, v, scale, causal=True)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], scale * (q[:, 0] * k[:, 0]).sum(-1), rtol=0, atol=1e-14)
    o_f, l_f = oracle.attention_reference(q, k, v, scale, causal=False)
    np.testing.assert_allclose(o[:, -1], o_f[:, -1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, -1], l_f[:, -1], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_sequence(causal):
    """N = 1, the smallest size the library accepts: the one weight is 1, so O is
    the value row and L is the one score, for the definition and the tiled form."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((4, 1, 12)) for _ in range(3))
    scale = 0.3
    want_l = scale * (q[:, 0] * k[:, 0]).sum(-1)
    for o, lse in (oracle.attention_reference(q, k, v, scale, causal),
                   oracle.attention_tiled(q, k, v, scale, causal, 16, 16)):
        np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, 0], want_l, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- invariants


def test_key_permutation_invariance():
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((30, 8)) for _ in range(3))
    perm = rng.permutation(30)
    o1, l1 = oracle.attention_reference(q, k, v, 0.4)
    o2, l2 = oracle.attention_reference(q, k[perm], v[perm], 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_per_row_score_shift():
    """Adding u to every key shifts row i's scores by scale*q_i.u: O unchanged,
    L shifted by exactly that amount (this pins the max/L bookkeeping)."""
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((25, 8)) for _ in range(3))
    u = rng.standard_normal(8) * 5
    scale = 0.35
    for causal in (False, True):
        o1, l1 = oracle.attention_reference(q, k, v, scale, causal)
        o2, l2 = oracle.attention_reference(q, k + u, v, scale, causal)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, scale * (q @ u), rtol=0, atol=1e-12)


def test_scale_folds_into_q():
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((2, 19, 8)) for _ in range(3))
    o1, l1 = oracle.attention_reference(q * 4.0, k, v, 0.125)
    o2, l2 = oracle.attention_reference(q, k, v, 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)


# ------------------------------------------------- tiled re-derivation and rows


# the FA2 tutorial's test shapes (ragged tails on both axes), square for causal
@pytest.mark.parametrize("n,d", [(128, 64), (100, 64), (37, 32), (200, 128), (1, 16), (300, 8)])
@pytest.mark.parametrize("bq,bk", [(16, 16), (7, 5), (None, None)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_equals_definition(n, d, bq, bk, causal):
    rng = np.random.default_rng(n * 31 + d)
    q, k, v = (rng.standard_normal((2, n, d)) * 2 for _ in range(3))
    bq = bq or n
    bk = bk or n
    scale = 1 / math.sqrt(d)
    o_n, l_n = oracle.attention_reference(q, k, v, scale, causal)
    o_t, l_t = oracle.attention_tiled(q, k, v, scale, causal, bq, bk)
    np.testing.assert_allclose(o_t, o_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_t, l_n, rtol=0, atol=1e-12)


def test_non_square_tiled_equals_definition():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((37, 32))
    k, v = rng.standard_normal((53, 32)), rng.standard_normal((53, 32))
    o_n, l_n = oracle.attention_reference(q, k, v, 0.2)
    o_t, l_t = oracle.attention_tiled(q, k, v, 0.2, bq=16, bk=16)
    np.testing.assert_allclose(o_t, o_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_t, l_n, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_full(causal):
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((3, 700, 16)) for _ in range(3))
    rows = inputs.sample_rows(700, 1, 3, count=64)
    assert all(r[0] == 0 and r[-1] == 699 and len(set(r)) == 64 for r in rows)
    o_f, l_f = oracle.attention_reference(q, k, v, 0.25, causal)
    o_r, l_r = oracle.attention_rows(q, k, v, rows, 0.25, causal)
    for h in range(3):
        np.testing.assert_allclose(o_r[h], o_f[h][rows[h]], rtol=0, atol=1e-14)
        np.testing.assert_allclose(l_r[h], l_f[h][rows[h]], rtol=0, atol=1e-14)


# ---------------------------------------------------------------- decoders


def test_e4m3_decoder_against_format_definition():
    dec = oracle.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    known = {
        0x00: 0.0, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x08: 2.0**-6, 0x30: 0.5,
        0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0,
        0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0,
    }
    for code, val in known.items():
        assert dec[code] == val, hex(code)
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert np.isnan(dec).sum() == 2
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0)  # strictly increasing over the finite codes
    np.testing.assert_array_equal(dec[0x80:0xFF], -pos)


def test_e4m3_decoder_against_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = oracle.e4m3_bits_to_f64(codes.numpy())
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(dec[ok], ref[ok])


def test_bf16_decoder_against_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(0)) * 100
    xb = x.to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(inputs.bits_u16(xb)), xb.double().numpy())


def test_quantiser_roundtrip_is_within_half_step():
    q, _, _ = inputs.make_qkv_f32(1, 1, 64, 32, seed=3)
    codes, ds = inputs.quantize_e4m3(q)
    back = oracle.dequantize(inputs.bits_u8(codes), "e4m3", ds)
    x = q.double().numpy()
    assert np.abs(back).max() <= 448 * ds * (1 + 1e-7)
    # e4m3 has 3 mantissa bits: relative error <= 2^-4 for normals
    big = np.abs(x) > ds * 2.0**-6 * 8
    assert np.all(np.abs(back - x)[big] <= np.abs(x)[big] * 2.0**-4 + 1e-12)


# ---------------------------------------------------------------- mutation check


def _mutant_no_scale(qrows, k, scale, keep):
    s = np.matmul(qrows, k.T)
    return np.where(keep, s, -np.inf) if keep is not None else s


def _mutant_sign(qrows, k, scale, keep):
    s = -float(scale) * np.matmul(qrows, k.T)
    return np.where(keep, s, -np.inf) if keep is not None else s


def _mutant_mask_strict(qrows, k, scale, keep):
    s = float(scale) * np.matmul(qrows, k.T)
    if keep is not None:
        keep = keep & ~np.eye(*keep.shape, dtype=bool)  # drops the diagonal key
        keep[0, 0] = True
    return np.where(keep, s, -np.inf) if keep is not None else s


@pytest.mark.parametrize("mutant", [_mutant_no_scale, _mutant_sign, _mutant_mask_strict])
def test_brute_force_pin_catches_planted_mistakes(monkeypatch, mutant):
    rng = np.random.default_rng(21)
    n, d = 6, 3
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    scale = 0.5
    causal = mutant is _mutant_mask_strict
    o_ref, l_ref = _mp_attention(q, k, v, scale, causal)
    monkeypatch.setattr(oracle_attention, "_scores", mutant)
    o, lse = oracle_attention.attention_reference(q, k, v, scale, causal)
    err = max(np.abs(o - o_ref).max(), np.abs(lse - l_ref).max())
    assert err > 1e-3
