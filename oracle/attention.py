"""Plain float64 attention forward: the definition, written out, and the
tile-by-tile online-softmax re-derivation.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Slow on purpose: no
blocking, fusion or reordering beyond what each cited passage states.  A matrix
product (``numpy.matmul``) serves as a step where the definition multiplies
matrices.

Shapes: ``q, k, v`` are float64 arrays ``[..., N, d]`` (any number of leading
batch/head axes; heads never interact).  Outputs are ``O [..., N, d]`` and the
per-row natural-log logsumexp ``L [..., N]``.
"""

from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# Decoding of the stored element formats into exact float64 values.
# --------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values.

    A bfloat16 is the upper 16 bits of an IEEE-754 binary32, so shifting the
    pattern into the top half of a 32-bit word gives the binary32 with the same
    value; widening binary32 -> binary64 is exact.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(bits) -> np.ndarray:
    """FP8 E4M3 ("fn": finite, no infinities) bit patterns (uint8) -> float64.

    Format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
    exponent field 0 encodes subnormals (m/8) * 2^-6; otherwise the value is
    (1 + m/8) * 2^(e-7).  The two patterns S.1111.111 (0x7F, 0xFF) are NaN, so
    the largest finite magnitude is 1.75 * 2^8 = 448.  Every value is exact in
    float64.
    """
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where((b & 0x80) != 0, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    subnormal = sign * (m / 8.0) * np.ldexp(1.0, -6)
    val = np.where(e == 0, subnormal, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, val)


def dequantize(codes, fmt: str, descale: float = 1.0) -> np.ndarray:
    """Stored codes -> float64 real values.

    ``fmt`` is ``"f32"`` (float32 array), ``"bf16"`` (uint16 bit patterns) or
    ``"e4m3"`` (uint8 bit patterns).  For e4m3 the real value is
    ``code_value * descale`` with a per-tensor descale: the FP8 page keeps one
    descale per tensor and head and folds it into the score scale
    ("Who am I, what's mine?"); one scalar per tensor is the special case used
    here.
    """
    if fmt == "f32":
        return np.asarray(codes, dtype=np.float32).astype(np.float64)
    if fmt == "bf16":
        return bf16_bits_to_f64(codes)
    if fmt == "e4m3":
        return e4m3_bits_to_f64(codes) * float(descale)
    raise ValueError(f"unknown format {fmt!r}")


# --------------------------------------------------------------------------
# The definition (materialised scores).
# --------------------------------------------------------------------------


def _causal_keep(n_q_rows: np.ndarray, n_keys: int) -> np.ndarray:
    """Boolean [len(rows), n_keys]: key j is kept for query row i iff j <= i.

    "FlashAttention-2 from PyTorch to Triton": the kernel keeps k_pos <= q_pos,
    and its tests build the reference mask with a lower-triangular ``tril``,
    causal only for square inputs.
    """
    return np.arange(n_keys)[None, :] <= np.asarray(n_q_rows)[:, None]


def _scores(qrows: np.ndarray, k: np.ndarray, scale: float, keep) -> np.ndarray:
    """S = scale * Q K^T for one head, masked keys set to -inf.

    A key excluded by the mask contributes exp(-inf) = 0 exactly, i.e. it is
    left out of the softmax, rather than given a large negative score.
    """
    s = float(scale) * np.matmul(qrows, k.T)
    if keep is not None:
        s = np.where(keep, s, -np.inf)
    return s


def attention_probs(q, k, scale: float, causal: bool = False) -> np.ndarray:
    """Row-softmax probabilities P = softmax(scale * Q K^T) for every head.

    "Kernels and Memory in LLM Inference", "Attention, said plainly again":
    compare every query with every key, subtract the row max, exponentiate,
    then normalise each row.  Returns P with shape [..., N, N].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    lead = q.shape[:-2]
    n, nk = q.shape[-2], k.shape[-2]
    qf = q.reshape((-1, n, q.shape[-1]))
    kf = k.reshape((-1, nk, k.shape[-1]))
    out = np.empty((qf.shape[0], n, nk))
    keep = _causal_keep(np.arange(n), nk) if causal else None
    for h in range(qf.shape[0]):
        s = _scores(qf[h], kf[h], scale, keep)
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m)
        out[h] = e / e.sum(axis=-1, keepdims=True)
    return out.reshape(lead + (n, nk))


def _attention_one_head(qrows, rows, k, v, scale, causal):
    """O and L for the given query rows of one head (materialised scores).

    For each row i:  m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i),
    O_i = sum_j exp(s_ij - m_i) v_j / l_i,  L_i = m_i + ln l_i
    ("FlashAttention-2 from PyTorch to Triton": L is the per-row logsumexp of
    the scaled scores, equal to log sum_k exp(S_ik) over the whole row).
    """
    keep = _causal_keep(rows, k.shape[0]) if causal else None
    s = _scores(qrows, k, scale, keep)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    o = np.matmul(e, v) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def attention_reference(q, k, v, scale: float, causal: bool = False):
    """Full attention forward in float64: returns (O [..., N, d], L [..., N]).

    The naive materialised form ("Kernels and Memory in LLM Inference", "The
    object in the middle is the problem": build S, softmax it, multiply by V),
    one head at a time so only one N x N score block is alive.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lead = q.shape[:-2]
    n, d = q.shape[-2], q.shape[-1]
    nk, dv = k.shape[-2], v.shape[-1]
    if causal and n != nk:
        raise ValueError("causal attention is defined here for square inputs only")
    qf, kf, vf = q.reshape(-1, n, d), k.reshape(-1, nk, d), v.reshape(-1, nk, dv)
    o = np.empty((qf.shape[0], n, dv))
    lse = np.empty((qf.shape[0], n))
    rows = np.arange(n)
    for h in range(qf.shape[0]):
        o[h], lse[h] = _attention_one_head(qf[h], rows, kf[h], vf[h], scale, causal)
    return o.reshape(lead + (n, dv)), lse.reshape(lead + (n,))


def attention_rows(q, k, v, rows, scale: float, causal: bool = False):
    """O and L of selected query rows only, for every head.

    ``q, k, v``: [BH, N, d]; ``rows``: int array [BH, R] (the rows of head h
    are ``rows[h]``).  Returns O [BH, R, d] and L [BH, R].  Same definition as
    :func:`attention_reference`; each row is independent of every other row,
    so computing a subset changes nothing.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    bh, r = rows.shape
    o = np.empty((bh, r, v.shape[-1]))
    lse = np.empty((bh, r))
    for h in range(bh):
        o[h], lse[h] = _attention_one_head(q[h][rows[h]], rows[h], k[h], v[h], scale, causal)
    return o, lse


# --------------------------------------------------------------------------
# Grouped-query attention: query heads share K/V heads.
# --------------------------------------------------------------------------


def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """The K/V head that query head ``h`` reads under grouped-query attention.

    "Kernels and Memory in LLM Inference", "Store less: MQA, GQA, MLA",
    "Grouped-query attention (2023)": the query heads are split into groups
    and each group gets one K/V head of its own; one group is multi-query
    attention, one group per head is ordinary multi-head attention.  The page
    does not say which query heads form a group; here a group is
    ``n_heads // n_kv_heads`` consecutive query heads, so group ``g`` (query
    heads ``g*G .. g*G + G - 1``) reads K/V head ``g``.
    """
    if n_kv_heads < 1 or n_heads % n_kv_heads != 0:
        raise ValueError(f"n_heads ({n_heads}) must be a multiple of n_kv_heads ({n_kv_heads})")
    if not 0 <= h < n_heads:
        raise ValueError(f"head {h} out of range")
    return h // (n_heads // n_kv_heads)


def attention_gqa(q, k, v, scale: float, causal: bool = False):
    """Grouped-query attention forward in float64.

    ``q``: [B, H, N, d]; ``k``, ``v``: [B, H_kv, N, d] with H a multiple of
    H_kv.  Query head h of batch b is ordinary attention
    (:func:`attention_reference`) against K/V head ``kv_head_of(h, H, H_kv)``
    of batch b.  Returns O [B, H, N, d] and L [B, H, N].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n, _ = q.shape
    hkv = k.shape[1]
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty((B, H, n))
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, hkv)
            o[b, h], lse[b, h] = attention_reference(q[b, h], k[b, g], v[b, g], scale, causal)
    return o, lse


def attention_gqa_rows(q, k, v, rows, scale: float, causal: bool = False):
    """Selected query rows of :func:`attention_gqa`.

    ``q``: [B, H, N, d]; ``k``, ``v``: [B, H_kv, N, d]; ``rows``: int array
    [B*H, R] (rows of query head (b, h) are ``rows[b*H + h]``).  Returns
    O [B*H, R, d] and L [B*H, R].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    B, H = q.shape[:2]
    hkv = k.shape[1]
    o = np.empty((B * H, rows.shape[1], v.shape[-1]))
    lse = np.empty((B * H, rows.shape[1]))
    for b in range(B):
        for h in range(H):
            g = kv_head_of(h, H, hkv)
            r = rows[b * H + h]
            o[b * H + h], lse[b * H + h] = _attention_one_head(q[b, h][r], r, k[b, g], v[b, g], scale, causal)
    return o, lse


# --------------------------------------------------------------------------
# Tile-by-tile online-softmax re-derivation (tiny inputs only).
# --------------------------------------------------------------------------


def attention_tiled(q, k, v, scale: float, causal: bool = False, bq: int = 16, bk: int = 16):
    """FlashAttention-2 forward, one query tile and one key tile at a time.

    Follows "FlashAttention-2 from PyTorch to Triton" (the FA2 forward pass and
    its PyTorch double loop), in float64, with ragged last tiles allowed:

    * per query tile: m = -inf, l = 0, O = 0 (unnormalised);
    * per key tile:   S = scale * Q_i K_j^T (masked keys -> -inf),
      m_new = max(m, rowmax S), P = exp(S - m_new), alpha = exp(m - m_new),
      l = alpha * l + rowsum P, O = alpha * O + P V_j, m = m_new
      (alpha multiplies the old state before the new tile is added -- the
      order the FP8 page insists on in "Online softmax, one strip at a time");
    * after the last key tile: O / l, and L = m + log l.

    On the first key tile alpha = exp(-inf - m_new) = 0, so no special case
    is needed.  Returns (O, L) like :func:`attention_reference`.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lead = q.shape[:-2]
    n, d = q.shape[-2], q.shape[-1]
    nk, dv = k.shape[-2], v.shape[-1]
    if causal and n != nk:
        raise ValueError("causal attention is defined here for square inputs only")
    qf, kf, vf = q.reshape(-1, n, d), k.reshape(-1, nk, d), v.reshape(-1, nk, dv)
    o_all = np.empty((qf.shape[0], n, dv))
    l_all = np.empty((qf.shape[0], n))
    with np.errstate(invalid="ignore"):
        for h in range(qf.shape[0]):
            for i0 in range(0, n, bq):
                rows = np.arange(i0, min(i0 + bq, n))
                qi = qf[h, rows]
                m_i = np.full((len(rows), 1), -np.inf)
                l_i = np.zeros((len(rows), 1))
                o_i = np.zeros((len(rows), dv))
                for j0 in range(0, nk, bk):
                    cols = np.arange(j0, min(j0 + bk, nk))
                    s = float(scale) * np.matmul(qi, kf[h, cols].T)
                    if causal:
                        s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
                    m_new = np.maximum(m_i, s.max(axis=-1, keepdims=True))
                    p = np.exp(s - m_new)
                    alpha = np.exp(m_i - m_new)
                    l_i = alpha * l_i + p.sum(axis=-1, keepdims=True)
                    o_i = alpha * o_i + np.matmul(p, vf[h, cols])
                    m_i = m_new
                o_all[h, rows] = o_i / l_i
                l_all[h, rows] = (m_i + np.log(l_i))[:, 0]
    return o_all.reshape(lead + (n, dv)), l_all.reshape(lead + (n,))


# --------------------------------------------------------------------------
# Backward pass: gradients of O with respect to Q, K and V.
# --------------------------------------------------------------------------


def attention_backward(q, k, v, do, scale: float, causal: bool = False):
    """dQ, dK, dV of the attention forward for the upstream gradient dO, float64.

    The pages name the ingredients of FlashAttention's backward ("FlashAttention-2
    from PyTorch to Triton", item 5 of the list of what the first kernel leaves
    out; "Kernels and Memory in LLM Inference", "Training detour (brief)"): the
    probabilities are rebuilt from L as P = exp(S - L), a row term
    D = rowsum(dO * O) is precomputed, dK and dV are built per key tile and dQ
    is accumulated.  The formulas themselves are the chain rule applied to the
    forward's definition (S = scale Q K^T with masked scores excluded,
    P = row softmax of S, O = P V):

        dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic (= sum_j P_ij dP_ij),
        dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.

    ``q, k, v, do``: [..., N, d].  Returns (dQ, dK, dV) with the input shapes.
    One head at a time; P is materialised (N x N), so N is kept small.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lead = q.shape[:-2]
    n, d = q.shape[-2], q.shape[-1]
    nk, dv = k.shape[-2], v.shape[-1]
    if causal and n != nk:
        raise ValueError("causal attention is defined here for square inputs only")
    qf, kf, vf, dof = q.reshape(-1, n, d), k.reshape(-1, nk, d), v.reshape(-1, nk, dv), do.reshape(-1, n, dv)
    dq, dk, dvv = np.empty_like(qf), np.empty_like(kf), np.empty_like(vf)
    keep = _causal_keep(np.arange(n), nk) if causal else None
    for h in range(qf.shape[0]):
        s = _scores(qf[h], kf[h], scale, keep)
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m)
        p = e / e.sum(axis=-1, keepdims=True)
        o = np.matmul(p, vf[h])
        dvv[h] = np.matmul(p.T, dof[h])
        dp = np.matmul(dof[h], vf[h].T)
        drow = (dof[h] * o).sum(axis=-1, keepdims=True)
        ds = p * (dp - drow)
        dq[h] = float(scale) * np.matmul(ds, kf[h])
        dk[h] = float(scale) * np.matmul(ds.T, qf[h])
    return dq.reshape(lead + (n, d)), dk.reshape(lead + (nk, d)), dvv.reshape(lead + (nk, dv))


def attention_backward_tiled(q, k, v, do, scale: float, causal: bool = False, bq: int = 16, bk: int = 16):
    """The same gradients in the tiled order the pages describe, float64.

    "FlashAttention-2 from PyTorch to Triton", item 5 of what the first kernel
    leaves out: with L from the forward and D = rowsum(dO * O) computed first,
    iterate over the query tiles for each key tile; per (key tile j, query
    tile i) rebuild P = exp(S - L) ("Kernels and Memory in LLM Inference",
    "Training detour (brief)": the attention tile is recomputed on chip when it
    is needed), add P^T dO_i to dV_j and scale dS^T Q_i to dK_j, and accumulate
    scale dS K_j into dQ_i.  Ragged last tiles are allowed.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lead = q.shape[:-2]
    n, d = q.shape[-2], q.shape[-1]
    nk, dv = k.shape[-2], v.shape[-1]
    o_all, l_all = attention_reference(q, k, v, scale, causal)
    qf, kf, vf, dof = q.reshape(-1, n, d), k.reshape(-1, nk, d), v.reshape(-1, nk, dv), do.reshape(-1, n, dv)
    of, lf = o_all.reshape(-1, n, dv), l_all.reshape(-1, n)
    dq, dk, dvv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for h in range(qf.shape[0]):
        drow = (dof[h] * of[h]).sum(axis=-1)
        for j0 in range(0, nk, bk):
            cols = np.arange(j0, min(j0 + bk, nk))
            for i0 in range(0, n, bq):
                rows = np.arange(i0, min(i0 + bq, n))
                s = float(scale) * np.matmul(qf[h, rows], kf[h, cols].T)
                p = np.exp(s - lf[h, rows][:, None])
                if causal:
                    p = np.where(cols[None, :] <= rows[:, None], p, 0.0)
                dvv[h, cols] += np.matmul(p.T, dof[h, rows])
                dp = np.matmul(dof[h, rows], vf[h, cols].T)
                ds = p * (dp - drow[rows][:, None])
                dk[h, cols] += float(scale) * np.matmul(ds.T, qf[h, rows])
                dq[h, rows] += float(scale) * np.matmul(ds, kf[h, cols])
    return dq.reshape(lead + (n, d)), dk.reshape(lead + (nk, d)), dvv.reshape(lead + (nk, dv))
