"""The allocation-free split-KV entry point, through the C ABI.

attn_fwd_split_noalloc is for callers that cannot allocate device memory when
they call the library (a plugin whose host application owns all device memory,
a loop that cannot afford cudaMalloc's synchronisation): its scratch is an
array the library declares in device memory.  This file checks, on two calls in
a row, that it returns exactly (bit for bit) what attn_fwd_split returns with a
caller-provided workspace -- the same kernels run on the same inputs with the
same split, so any difference would mean the shared array was misused -- and
that it refuses sizes its fixed array cannot hold.  It is named
to be collected last, so a run that stops at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""

import pytest
import torch

from tiled_attention_fa2_gb300 import binding

from parity import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(built_library):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return binding.load_library()


def _no_alloc(lib, dev, case, n_splits, o, lse):
    ds = case.descales if case.dtype == "e4m3" else (1.0, 1.0, 1.0)
    code = 2 if case.dtype == "e4m3" else 1
    return lib.attn_fwd_split_noalloc(dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), case.B, case.H, case.N, case.d, case.scale, ds[0], ds[1],
                                      ds[2], 0, code, n_splits, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,d,n_splits", [("bf16", 128, 4), ("bf16", 64, 0), ("e4m3", 128, 3)])
def test_no_alloc_entry_matches_workspace_entry_on_two_calls(lib, dtype, d, n_splits):
    for call in range(2):
        case = make_case(1, 2, 3000, d, dtype, seed=40 + call)
        dev = [t.cuda() for t in case.stored]
        ds = case.descales if dtype == "e4m3" else None
        o_ref, l_ref = binding.attn_fwd_split(*dev, n_splits=n_splits, descales=ds, scale=case.scale)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(l_ref)
        assert _no_alloc(lib, dev, case, n_splits, o, lse) == 0, lib.attn_last_error()
        torch.cuda.synchronize()
        assert binding.get_device_status() == 0
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, l_ref)


def test_no_alloc_entry_refuses_sizes_beyond_its_scratch(lib):
    # 8 ranges x 65536 rows x 128 features x 4 bytes = 256 MiB of partial O.
    # The buffers have the declared shape (16 MiB each), so even a call that
    # wrongly went ahead would stay inside them.
    B, H, N, d = 1, 8, 8192, 128
    q, k, v, o = (torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = lib.attn_fwd_split_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                    N, d, 0.1, 1.0, 1.0, 1.0, 0, 1, 8, torch.cuda.current_stream().cuda_stream)
    assert st == 2
    assert b"64 MiB" in lib.attn_last_error()
