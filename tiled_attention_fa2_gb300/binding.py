"""ctypes binding of libattn_fa2.so (declared in include/attn_fa2.h).

Argument marshalling only: torch tensors provide device memory and the CUDA
stream; every step of the attention forward runs in the library's kernels.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libattn_fa2.so")

ATTN_F32, ATTN_BF16, ATTN_E4M3 = 0, 1, 2
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_MISALIGNED",
                4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT"}

# Every symbol include/attn_fa2.h declares, with its ctypes signature.
_VP, _I, _F, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
SIGNATURES = {
    "attn_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _I, _I, _VP]),
    "attn_fwd_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _F, _F, _F, _I, _VP]),
    "attn_fwd_gqa": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, _F, _F, _F, _I, _I, _VP]),
    "attn_fwd_host": (_I, [_VP] * 10 + [_I, _I, _I, _I, _F, _F, _F, _F, _I, _I, _VP]),
    "attn_get_device_status": (_I, [_VP]),
    "attn_set_wait_limit_ns": (_U64, [_U64]),
    "attn_set_poly_exp2": (_I, [_I]),
    "attn_selftest_wait_timeout": (_I, [_U64, _VP]),
    "attn_fwd_split_plan": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]),
    "attn_fwd_split": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _F, _F, _F, _I, _I, _I, _VP, ctypes.c_size_t,
                            _VP]),
    "attn_fwd_split_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _F, _F, _F, _I, _I, _I, _VP]),
    "attn_bwd_workspace_size": (_I, [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "attn_bwd": (_I, [_VP] * 10 + [ctypes.c_size_t, _I, _I, _I, _I, _F, _I, _VP]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_last_error": (ctypes.c_char_p, []),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} not found: build it with `python -m tiled_attention_fa2_gb300._build` "
                              "(or __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int):
    if status != 0:
        lib = load_library()
        raise AttnError(status, lib.attn_last_error().decode() or lib.attn_status_string(status).decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return ATTN_E4M3
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _shape(q, k, v):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"q, k, v must share one [B, H, N, d] shape (got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)})")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must have the same dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if k.device != q.device or v.device != q.device:
        raise ValueError(f"q, k, v must be on one device (got {q.device}, {k.device}, {v.device})")
    return tuple(int(x) for x in q.shape)


def _require(name, t, device, dtype, shape):
    """A buffer the library reads or writes: a contiguous CUDA tensor of the
    given dtype and shape on `device` (a host tensor here would hand the kernel
    a host address)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"(got {t.dtype} {tuple(t.shape)})")


def _outputs(q, o, lse, B, H, N, d, code):
    odt = torch.float32 if code == ATTN_F32 else torch.bfloat16
    if o is None:
        o = torch.empty((B, H, N, d), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _require("o", o, q.device, odt, (B, H, N, d))
    _require("lse", lse, q.device, torch.float32, (B, H, N))
    return o, lse


def attn_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """Attention forward on CUDA tensors [B, H, N, d] (float32, bfloat16, or
    e4m3 codes with unit descales).  Returns (o, lse)."""
    B, H, N, d = _shape(q, k, v)
    code = _dtype_code(q)
    o, lse = _outputs(q, o, lse, B, H, N, d, code)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                            scale, int(bool(causal)), code, _stream_handle(stream, q.device)))
    return o, lse


def attn_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o=None, lse=None, scale=None, causal=False,
                 stream=None):
    """FP8 E4M3 forward (uint8 or float8_e4m3fn CUDA tensors) with per-tensor
    descales; bf16 O, fp32 L.  Returns (o, lse)."""
    B, H, N, d = _shape(q, k, v)
    if _dtype_code(q) != ATTN_E4M3:
        raise TypeError("attn_fwd_fp8 takes e4m3 codes (uint8 or float8_e4m3fn)")
    o, lse = _outputs(q, o, lse, B, H, N, d, ATTN_E4M3)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                d, scale, float(q_descale), float(k_descale), float(v_descale), int(bool(causal)),
                                _stream_handle(stream, q.device)))
    return o, lse


def attn_fwd_gqa(q, k, v, descales=None, o=None, lse=None, scale=None, causal=False, stream=None):
    """Grouped-query attention forward: q [B, H, N, d]; k, v [B, H_kv, N, d]
    with H a multiple of H_kv (query head h reads K/V head h // (H // H_kv)).
    float32, bfloat16, or e4m3 codes with ``descales`` = (q, k, v) descales.
    Returns (o [B, H, N, d], lse [B, H, N])."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError(f"q must be [B, H, N, d] and k, v one [B, H_kv, N, d] shape (got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)})")
    B, H, N, d = (int(x) for x in q.shape)
    Hkv = int(k.shape[1])
    if (int(k.shape[0]), int(k.shape[2]), int(k.shape[3])) != (B, N, d):
        raise ValueError(f"k, v must be [{B}, H_kv, {N}, {d}] (got {tuple(k.shape)})")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must have the same dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.device != q.device:
            raise ValueError("q, k, v must be contiguous CUDA tensors on one device")
    code = _dtype_code(q)
    o, lse = _outputs(q, o, lse, B, H, N, d, code)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ds = tuple(float(x) for x in descales) if descales is not None else (1.0, 1.0, 1.0)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.attn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv,
                                N, d, scale, ds[0], ds[1], ds[2], int(bool(causal)), code,
                                _stream_handle(stream, q.device)))
    return o, lse


def attn_fwd_host(h_q, h_k, h_v, h_o, h_lse, d_q, d_k, d_v, d_o, d_lse, scale=None, causal=False,
                  descales=(1.0, 1.0, 1.0), stream=None):
    """End-to-end forward from (page-locked) host tensors through caller-owned
    device staging tensors: H2D copies, forward, D2H copies, all enqueued on
    `stream`.  The caller synchronises before reading h_o / h_lse."""
    if h_q.dim() != 4:
        raise ValueError(f"h_q must be [B, H, N, d] (got shape {tuple(h_q.shape)})")
    B, H, N, d = (int(x) for x in h_q.shape)
    code = _dtype_code(h_q)
    odt = torch.float32 if code == ATTN_F32 else torch.bfloat16
    # Every copy moves the bytes of [B, H, N, d] (or [B, H, N]) elements, so each
    # buffer must hold exactly that many of its dtype.
    want = {"h_q": (h_q, h_q.dtype, (B, H, N, d)), "h_k": (h_k, h_q.dtype, (B, H, N, d)),
            "h_v": (h_v, h_q.dtype, (B, H, N, d)), "h_o": (h_o, odt, (B, H, N, d)),
            "h_lse": (h_lse, torch.float32, (B, H, N))}
    for name, (t, dt, shape) in want.items():
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
        if t.dtype != dt or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a {dt} tensor of shape {shape} (got {t.dtype} {tuple(t.shape)})")
    if not isinstance(d_q, torch.Tensor) or not d_q.is_cuda:
        raise ValueError("d_q must be a CUDA tensor")
    dev = d_q.device
    for name, t in (("d_q", d_q), ("d_k", d_k), ("d_v", d_v)):
        _require(name, t, dev, h_q.dtype, (B, H, N, d))
    _require("d_o", d_o, dev, odt, (B, H, N, d))
    _require("d_lse", d_lse, dev, torch.float32, (B, H, N))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = load_library()
    with torch.cuda.device(dev):
        _check(lib.attn_fwd_host(h_q.data_ptr(), h_k.data_ptr(), h_v.data_ptr(), h_o.data_ptr(), h_lse.data_ptr(),
                                 d_q.data_ptr(), d_k.data_ptr(), d_v.data_ptr(), d_o.data_ptr(), d_lse.data_ptr(),
                                 B, H, N, d, scale, float(descales[0]), float(descales[1]), float(descales[2]),
                                 int(bool(causal)), code, _stream_handle(stream, dev)))


def split_plan(B, H, N, d, n_splits=0):
    """(resolved split count, workspace bytes) of attn_fwd_split for these sizes."""
    lib = load_library()
    s = ctypes.c_int(0)
    nb = ctypes.c_size_t(0)
    _check(lib.attn_fwd_split_plan(int(B), int(H), int(N), int(d), int(n_splits), ctypes.byref(s), ctypes.byref(nb)))
    return s.value, nb.value


def attn_fwd_split(q, k, v, n_splits=0, descales=None, o=None, lse=None, scale=None, workspace=None, stream=None):
    """Non-causal split-KV forward (bf16, or e4m3 codes with `descales`).
    Allocates the workspace with torch unless one is given.  Returns (o, lse)."""
    B, H, N, d = _shape(q, k, v)
    code = _dtype_code(q)
    o, lse = _outputs(q, o, lse, B, H, N, d, code)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(q.device):
        _, nbytes = split_plan(B, H, N, d, n_splits)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {q.device}")
    ds = descales if descales is not None else (1.0, 1.0, 1.0)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.attn_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N,
                                  d, scale, float(ds[0]), float(ds[1]), float(ds[2]), 0, code, int(n_splits),
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, q.device)))
    return o, lse


def bwd_workspace_size(B, H, N, d) -> int:
    """Bytes of device workspace attn_bwd needs for these sizes."""
    nb = ctypes.c_size_t(0)
    _check(load_library().attn_bwd_workspace_size(int(B), int(H), int(N), int(d), ctypes.byref(nb)))
    return nb.value


def attn_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, scale=None, causal=False, workspace=None,
             stream=None):
    """Backward of the bf16 forward: (dq, dk, dv) for the upstream gradient dout.
    `o` and `lse` are the forward's outputs.  Allocates outputs and workspace
    with torch unless given."""
    B, H, N, d = _shape(q, k, v)
    if q.dtype != torch.bfloat16:
        raise TypeError("attn_bwd takes bfloat16 q, k, v")
    shape = (B, H, N, d)
    _require("o", o, q.device, torch.bfloat16, shape)
    _require("dout", dout, q.device, torch.bfloat16, shape)
    _require("lse", lse, q.device, torch.float32, (B, H, N))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _require(name, t, q.device, torch.bfloat16, shape)
    nbytes = bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {q.device}")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = load_library()
    with torch.cuda.device(q.device):
        _check(lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), B, H, N, d, scale, int(bool(causal)),
                            _stream_handle(stream, q.device)))
    return dq, dk, dv


def get_device_status(stream=None) -> int:
    """Synchronise and return the device status (0 = ok, 5 = a wait timed out)."""
    lib = load_library()
    return int(lib.attn_get_device_status(_stream_handle(stream, None)))


def selftest_wait_timeout(limit_ns: int = 10_000_000, stream=None) -> None:
    """Enqueue the bounded-wait self-test (see include/attn_fa2.h)."""
    lib = load_library()
    _check(lib.attn_selftest_wait_timeout(int(limit_ns), _stream_handle(stream, None)))


def set_wait_limit_ns(ns: int) -> int:
    return int(load_library().attn_set_wait_limit_ns(int(ns)))


def forward(q, k, v, causal=False, scale=None, descales=None):
    """Convenience: dispatch on dtype (e4m3 needs `descales`)."""
    if _dtype_code(q) == ATTN_E4M3 and descales is not None:
        return attn_fwd_fp8(q, k, v, *descales, scale=scale, causal=causal)
    return attn_fwd(q, k, v, scale=scale, causal=causal)


def set_poly_exp2(on: bool) -> bool:
    """Split exponential for the e4m3 forward (one exponential pair in four by a
    polynomial on the FMA pipe); returns the previous setting."""
    prev = load_library().attn_set_poly_exp2(int(bool(on)))
    if prev < 0:
        raise ValueError("attn_set_poly_exp2 refused the setting")
    return bool(prev)
