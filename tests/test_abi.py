"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/attn_fa2.h declares, and rejects invalid arguments
before anything reaches CUDA."""

import ctypes
import os
import re

import pytest

from tiled_attention_fa2_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fa2.h")


@pytest.fixture(scope="module")
def lib(built_library):
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_fp8", "attn_fwd_host", "attn_get_device_status",
            "attn_status_string", "attn_last_error", "attn_set_wait_limit_ns",
            "attn_selftest_wait_timeout"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(binding.SIGNATURES)


def test_status_strings(lib):
    assert lib.attn_status_string(0) == b"ok"
    assert lib.attn_status_string(5) == b"device wait timed out"
    assert lib.attn_status_string(99) == b"unknown status"


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced on these paths


def call_fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, N=256, d=64, scale=0.125, causal=0, dtype=1,
             stream=None)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"], a["scale"],
                        a["causal"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(scale=-1.0), 1),
    (dict(causal=2), 1), (dict(dtype=7), 1),
    (dict(d=96), 2), (dict(d=32), 2), (dict(dtype=2, d=64), 2), (dict(dtype=0, d=48), 2),
    (dict(q=FAKE + 8), 3), (dict(o=FAKE + 4), 3), (dict(o=FAKE + 16), 3), (dict(lse=FAKE + 2), 3),
    (dict(B=65536, H=65536), 1),
])
def test_invalid_arguments_are_rejected_on_the_host(lib, kw, status):
    assert call_fwd(lib, **kw) == status
    assert lib.attn_last_error() != b""


def test_fp8_descales_are_validated(lib):
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        st = lib.attn_fwd_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 0.1, bad, 1.0, 1.0, 0, None)
        assert st == 1


def test_host_entry_validates_before_copying(lib):
    st = lib.attn_fwd_host(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                           1, 1, 128, 64, 0.1, 1.0, 1.0, 1.0, 0, 1, None)
    assert st == 1
    st = lib.attn_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                           1, 1, 128, 64, 0.1, 1.0, 1.0, 1.0, 0, 9, None)
    assert st == 1
    # What only the kernel of the dtype requires is checked before the copies
    # too: an unsupported head dimension or an o that the bf16 kernel cannot
    # store to (32-byte rule) returns its own status, not a failed copy.
    for d, dtype, d_o, want in ((96, 1, FAKE, 2), (64, 2, FAKE, 2), (48, 0, FAKE, 2), (128, 1, FAKE + 16, 3)):
        st = lib.attn_fwd_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, d_o, FAKE,
                               1, 1, 128, d, 0.1, 1.0, 1.0, 1.0, 0, dtype, None)
        assert st == want, (d, dtype, st, lib.attn_last_error())


def test_wait_limit_setter_round_trips(lib):
    old = lib.attn_set_wait_limit_ns(5_000_000_000)
    assert lib.attn_set_wait_limit_ns(old) == 5_000_000_000
    assert lib.attn_set_wait_limit_ns(10) == old
    assert lib.attn_set_wait_limit_ns(old) == 1_000_000  # clamped to >= 1 ms


def test_binding_raises_when_library_is_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(ImportError):
        binding.load_library(str(tmp_path / "missing.so"))


def test_selftest_limit_is_validated_on_the_host(lib):
    assert lib.attn_selftest_wait_timeout(999_999, None) == 1


def test_split_plan_arithmetic(lib):
    import ctypes
    s = ctypes.c_int(0)
    nb = ctypes.c_size_t(0)
    # N = 1000 -> 8 key tiles; 3 requested -> 3 tiles per range -> 3 ranges
    assert lib.attn_fwd_split_plan(1, 2, 1000, 128, 3, ctypes.byref(s), ctypes.byref(nb)) == 0
    assert s.value == 3
    rows = 1 * 2 * 1000
    o_bytes = (3 * rows * 128 * 4 + 255) // 256 * 256
    assert nb.value == o_bytes + 3 * rows * 4
    # 6 requested over 8 tiles -> 2 tiles per range -> 4 ranges (no empty range)
    assert lib.attn_fwd_split_plan(1, 2, 1000, 128, 6, ctypes.byref(s), None) == 0
    assert s.value == 4
    # never more ranges than key tiles; one range needs no workspace
    assert lib.attn_fwd_split_plan(1, 1, 100, 64, 9, ctypes.byref(s), ctypes.byref(nb)) == 0
    assert s.value == 1 and nb.value == 0
    assert lib.attn_fwd_split_plan(0, 1, 100, 64, 2, None, None) == 1
    assert lib.attn_fwd_split_plan(1, 1, 100, 96, 2, None, None) == 1  # d must be 64 or 128
    assert lib.attn_fwd_split_plan(1, 1, 100, 64, -1, None, None) == 1


def call_split(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, N=1000, d=128, scale=0.1, qd=1.0, kd=1.0, vd=1.0,
             causal=0, dtype=1, n_splits=4, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return lib.attn_fwd_split(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"], a["scale"],
                              a["qd"], a["kd"], a["vd"], a["causal"], a["dtype"], a["n_splits"], a["ws"], a["wsb"],
                              None)


@pytest.mark.parametrize("kw,status", [
    (dict(causal=1), 2), (dict(dtype=0, d=64), 2), (dict(ws=None), 1), (dict(wsb=1024), 1),
    (dict(ws=FAKE + 16), 3), (dict(dtype=2, qd=0.0), 1), (dict(n_splits=-2), 1), (dict(q=None), 1),
])
def test_split_entry_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert call_split(lib, **kw) == status


def call_bwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE, wsb=1 << 40,
             B=1, H=2, N=256, d=128, scale=0.1, causal=0)
    a.update(kw)
    return lib.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["ws"],
                        a["wsb"], a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(dout=None), 1), (dict(dv=None), 1), (dict(ws=None), 1), (dict(N=0), 1),
    (dict(causal=3), 1), (dict(scale=0.0), 1), (dict(wsb=1024), 1), (dict(d=96), 2), (dict(d=32), 2),
    (dict(dq=FAKE + 8), 3), (dict(dout=FAKE + 4), 3), (dict(ws=FAKE + 16), 3), (dict(B=300, H=300, N=8), 2),
    # the preparation kernel reads o and dout 16 bytes at a time
    (dict(o=FAKE + 8), 3), (dict(dout=FAKE + 8), 3),
])
def test_backward_entry_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert call_bwd(lib, **kw) == status
    assert lib.attn_last_error() != b""


def test_backward_workspace_size(lib):
    # fp32 dQ accumulator (rows x d), then two fp32 vectors with one entry per row of
    # each head padded to a multiple of 128 rows, each rounded up to 256 bytes.
    for B, H, N, d in [(1, 1, 1, 64), (2, 3, 300, 128), (4, 16, 2048, 128)]:
        rows = B * H * N
        prows = B * H * (-(-N // 128) * 128)
        want = -(-rows * d * 4 // 256) * 256 + 2 * (-(-prows * 4 // 256) * 256)
        assert binding.bwd_workspace_size(B, H, N, d) == want
    with pytest.raises(binding.AttnError):
        binding.bwd_workspace_size(1, 1, 16, 96)


def call_gqa(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=8, Hkv=2, N=256, d=128, scale=0.1, qd=1.0, kd=1.0,
             vd=1.0, causal=0, dtype=1)
    a.update(kw)
    return lib.attn_fwd_gqa(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["N"], a["d"],
                            a["scale"], a["qd"], a["kd"], a["vd"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hkv=0), 1), (dict(Hkv=3), 1), (dict(Hkv=16), 1), (dict(H=0), 1), (dict(Hkv=-2), 1),
    (dict(q=None), 1), (dict(dtype=2, kd=0.0), 1), (dict(dtype=2, vd=float("nan")), 1), (dict(d=96), 2),
    (dict(k=FAKE + 8), 3), (dict(causal=2), 1),
])
def test_gqa_entry_rejects_bad_arguments_on_the_host(lib, kw, status):
    assert call_gqa(lib, **kw) == status
    assert lib.attn_last_error() != b""


def test_gqa_descales_are_ignored_for_bf16(lib):
    # Only an ATTN_E4M3 call reads the descales; a bf16 call with zero descales
    # passes validation and fails only on the (deliberately) unsupported d.
    assert call_gqa(lib, dtype=1, qd=0.0, kd=0.0, vd=0.0, d=96) == 2


def test_poly_exp2_setter_round_trips(lib):
    prev = lib.attn_set_poly_exp2(1)
    assert prev in (0, 1)
    assert lib.attn_set_poly_exp2(0) == 1
    assert lib.attn_set_poly_exp2(7) == -1  # refused, nothing changed
    assert lib.attn_set_poly_exp2(prev) == 0
