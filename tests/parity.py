"""Shared helpers of the GPU parity tests: seeded inputs, one GPU call
through the C ABI, and the float64 oracle on the same bytes.

The oracle always receives the stored codes (float32 values, bf16 bit
patterns, or e4m3 bytes with their descales) and decodes them itself.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import oracle
from tiled_attention_fa2_gb300 import binding, inputs

# Tolerances (max-abs over every compared element).
TOL_O = {"f32": 2e-2, "bf16": 2e-2, "e4m3": 6e-2}
TOL_L = {"f32": 1e-3, "bf16": 1e-3, "e4m3": 1e-3}
# The fp32 kernel is exact FFMA with an accurate exp2: a much tighter self-check.
TOL_F32_TIGHT = 1e-4


@dataclass
class Case:
    B: int
    H: int
    N: int
    d: int
    dtype: str                  # "f32" | "bf16" | "e4m3"
    stored: tuple               # CPU tensors handed to the GPU (q, k, v)
    codes: tuple                # numpy arrays handed to the oracle ([BH, N, d] each)
    descales: tuple = (1.0, 1.0, 1.0)
    scale_override: float | None = None  # softmax scale other than 1/sqrt(d)
    Hkv: int | None = None      # K/V heads (grouped-query attention); None = H

    @property
    def scale(self):
        return self.scale_override if self.scale_override is not None else 1.0 / math.sqrt(self.d)


def make_case(B, H, N, d, dtype, seed=0, q_mult=1.0, n_kv_heads=None) -> Case:
    """Seeded inputs; ``codes`` are [heads, N, d] per tensor (K and V have
    B * n_kv_heads heads under grouped-query attention)."""
    q, k, v = inputs.make_qkv_f32(B, H, N, d, seed=seed, q_mult=q_mult, n_kv_heads=n_kv_heads)
    hkv = None if n_kv_heads is None or n_kv_heads == H else int(n_kv_heads)
    shape = (-1, N, d)
    if dtype == "f32":
        stored = (q, k, v)
        codes = tuple(t.reshape(shape).numpy() for t in stored)
        return Case(B, H, N, d, dtype, stored, codes, Hkv=hkv)
    if dtype == "bf16":
        stored = tuple(inputs.to_bf16(t) for t in (q, k, v))
        codes = tuple(inputs.bits_u16(t).reshape(shape) for t in stored)
        return Case(B, H, N, d, dtype, stored, codes, Hkv=hkv)
    if dtype == "e4m3":
        qc, qd = inputs.quantize_e4m3(q)
        kc, kd = inputs.quantize_e4m3(k)
        vc, vd = inputs.quantize_e4m3(v)
        stored = (qc, kc, vc)
        codes = tuple(inputs.bits_u8(t).reshape(shape) for t in stored)
        return Case(B, H, N, d, dtype, stored, codes, (qd, kd, vd), Hkv=hkv)
    raise ValueError(dtype)


def run_gpu(case: Case, causal: bool):
    """One forward through the C ABI; returns (O float64 [BH,N,d], L float64 [BH,N])."""
    dev = [t.cuda() for t in case.stored]
    if case.Hkv is not None:
        o, lse = binding.attn_fwd_gqa(*dev, descales=case.descales, scale=case.scale, causal=causal)
    elif case.dtype == "e4m3":
        o, lse = binding.attn_fwd_fp8(*dev, *case.descales, scale=case.scale, causal=causal)
    else:
        o, lse = binding.attn_fwd(*dev, scale=case.scale, causal=causal)
    torch.cuda.synchronize()
    st = binding.get_device_status()
    assert st == 0, f"device status {st}"
    BH = case.B * case.H
    return (o.double().cpu().numpy().reshape(BH, case.N, case.d),
            lse.double().cpu().numpy().reshape(BH, case.N))


def _head(case: Case, h: int):
    """Query head h (over B*H) and the K/V head it reads, decoded by the oracle."""
    fmt = case.dtype
    hk = h
    if case.Hkv is not None:
        b, hq = divmod(h, case.H)
        hk = b * case.Hkv + oracle.kv_head_of(hq, case.H, case.Hkv)
    return tuple(oracle.dequantize(c[i], fmt, ds) for c, ds, i in zip(case.codes, case.descales, (h, hk, hk)))


def oracle_full(case: Case, causal: bool):
    BH = case.B * case.H
    o = np.empty((BH, case.N, case.d))
    lse = np.empty((BH, case.N))
    for h in range(BH):
        q, k, v = _head(case, h)
        o[h], lse[h] = oracle.attention_reference(q, k, v, case.scale, causal)
    return o, lse


def oracle_rows(case: Case, causal: bool, rows: np.ndarray):
    BH = case.B * case.H
    o = np.empty((BH, rows.shape[1], case.d))
    lse = np.empty((BH, rows.shape[1]))
    for h in range(BH):
        q, k, v = _head(case, h)
        oh, lh = oracle.attention_rows(q[None], k[None], v[None], rows[h][None], case.scale, causal)
        o[h], lse[h] = oh[0], lh[0]
    return o, lse


# Measured errors of every compared case, written as JSON at the end of the
# session when ATTN_PARITY_REPORT names a file (see tests/conftest.py).
REPORT = []


def errors(o_gpu, l_gpu, o_ref, l_ref, label=None):
    assert np.isfinite(o_gpu).all() and np.isfinite(l_gpu).all(), "non-finite GPU output"
    eo, el = float(np.abs(o_gpu - o_ref).max()), float(np.abs(l_gpu - l_ref).max())
    if label is not None:
        REPORT.append({"case": label, "o_max_abs": eo, "l_max_abs": el, "compared": int(o_ref.size)})
    return eo, el
