"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the
oracle's callers.

This module holds none of the attention arithmetic: it draws i.i.d. normal
Q/K/V, casts them to the stored element type, quantises them to FP8 with a
per-tensor absmax scale, and picks the sampled query rows that the largest
workloads are checked on.  The same bytes go to the GPU and to the oracle.

Recipe (one documented reading of "i.i.d. N(0,1) from seed 0"):
``torch.Generator('cpu').manual_seed(seed)``, then ``torch.randn`` of shape
[B, H, N, d] in float32 for Q, then K, then V, in that order; an optional
power-of-two multiplier on Q (exact) makes the row max move between key tiles.
"""

from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0  # largest finite magnitude of FP8 E4M3 ("fn" variant)


def make_qkv_f32(B: int, H: int, N: int, d: int, seed: int = 0, q_mult: float = 1.0, n_kv_heads: int | None = None):
    """Float32 Q, K, V drawn i.i.d. N(0, 1) on the CPU, in the order Q, K, V.

    Q is [B, H, N, d]; K and V are [B, n_kv_heads, N, d] (default H heads; fewer
    for grouped-query attention)."""
    hkv = H if n_kv_heads is None else int(n_kv_heads)
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, H, N, d), dtype=torch.float32, generator=g)
    k = torch.randn((B, hkv, N, d), dtype=torch.float32, generator=g)
    v = torch.randn((B, hkv, N, d), dtype=torch.float32, generator=g)
    if q_mult != 1.0:
        q = q * float(q_mult)
    return q, k, v


def make_dout_f32(B: int, H: int, N: int, d: int, seed: int = 0):
    """Float32 upstream gradient dO for the backward, i.i.d. N(0, 1) from
    ``torch.Generator('cpu').manual_seed(seed)`` (same recipe as Q, K, V)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn((B, H, N, d), dtype=torch.float32, generator=g)


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even cast to bfloat16 (torch's cast)."""
    return x.to(torch.bfloat16)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor absmax quantisation to FP8 E4M3.

    descale = absmax(x) / 448; codes = e4m3(x / descale) with round-to-nearest
    and saturation at +-448.  Returns (uint8 codes tensor, descale as a Python
    float holding a float32 value).  The real value of code c is
    ``e4m3(c) * descale``.
    """
    amax = float(x.abs().max())
    descale = np.float32(amax / E4M3_MAX) if amax > 0 else np.float32(1.0)
    y = (x / torch.tensor(descale, dtype=torch.float32)).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, float(descale)


def bits_u16(x_bf16: torch.Tensor) -> np.ndarray:
    """The bit patterns of a bfloat16 tensor as a numpy uint16 array."""
    return x_bf16.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_u8(codes: torch.Tensor) -> np.ndarray:
    """The bytes of a uint8 code tensor as a numpy uint8 array."""
    return codes.contiguous().numpy().view(np.uint8)


def sample_rows(N: int, B: int, H: int, count: int = 512) -> np.ndarray:
    """Seeded query rows checked per head on the largest workloads.

    For head (b, h): rows {0, N-1} plus ``count - 2`` distinct others drawn
    with ``numpy.random.default_rng(1000 + b*H + h)``, sorted.  Returns an
    int64 array [B*H, count] (all rows when N <= count).
    """
    out = []
    for b in range(B):
        for h in range(H):
            if N <= count:
                out.append(np.arange(N, dtype=np.int64))
                continue
            rng = np.random.default_rng(1000 + b * H + h)
            inner = rng.choice(np.arange(1, N - 1), size=count - 2, replace=False)
            out.append(np.sort(np.concatenate([[0, N - 1], inner]).astype(np.int64)))
    return np.stack(out)


# Named workloads: the sizes and element types the library is checked and
# measured on.  ``name -> dict(B, H, N, d, dtype, causal, q_mult[, Hkv])``;
# ``Hkv`` (K/V heads, grouped-query attention) defaults to H.
WORKLOADS = {
    "tiny_f32": dict(B=1, H=2, N=256, d=64, dtype="f32", causal=False, q_mult=1.0),
    "prefill_causal_bf16": dict(B=4, H=16, N=2048, d=128, dtype="bf16", causal=True, q_mult=1.0),
    "sweep_d64_bf16": dict(B=2, H=32, N=4096, d=64, dtype="bf16", causal=False, q_mult=1.0),
    "sweep_d128_bf16": dict(B=2, H=32, N=4096, d=128, dtype="bf16", causal=False, q_mult=1.0),
    "sweep_d128_bf16_qx8": dict(B=2, H=32, N=4096, d=128, dtype="bf16", causal=False, q_mult=8.0),
    "sweep_d64_bf16_qx8": dict(B=2, H=32, N=4096, d=64, dtype="bf16", causal=False, q_mult=8.0),
    "dit_e4m3": dict(B=1, H=56, N=30272, d=128, dtype="e4m3", causal=False, q_mult=1.0),
    "long_causal_bf16": dict(B=1, H=8, N=32768, d=128, dtype="bf16", causal=True, q_mult=1.0),
    "long_causal_e4m3": dict(B=1, H=8, N=32768, d=128, dtype="e4m3", causal=True, q_mult=1.0),
    # The DiT shape on 16 of its 56 heads: the small case whole-kernel profiles
    # are taken on (inputs still larger than L2, a quarter of the run time).
    "dit_e4m3_16h": dict(B=1, H=16, N=30272, d=128, dtype="e4m3", causal=False, q_mult=1.0),
    # Grouped-query attention at the head counts of a Llama-3-70B-class model
    # (64 query heads sharing 8 K/V heads, d = 128), causal prefill of 8192 tokens.
    "prefill_gqa_bf16": dict(B=1, H=64, Hkv=8, N=8192, d=128, dtype="bf16", causal=True, q_mult=1.0),
    "prefill_gqa_e4m3": dict(B=1, H=64, Hkv=8, N=8192, d=128, dtype="e4m3", causal=True, q_mult=1.0),
}


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of one forward: two N x N x d products per head
    (4 * B * H * N^2 * d), halved for causal (the counting convention of the
    bench harness in "FlashAttention-2 from PyTorch to Triton")."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f
