"""The Python binding refuses buffers the kernels cannot use, before any call
into the library: a host tensor where a device buffer is expected (the kernel
would be handed a host address), a wrong shape or dtype (a copy or a store
would run past the buffer).  Each case raises ValueError and launches nothing.
"""

import pytest
import torch

from tiled_attention_fa2_gb300 import binding

from parity import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev_case(built_library):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load_library()
    case = make_case(1, 2, 256, 128, "bf16", seed=3)
    return case, [t.cuda() for t in case.stored]


def test_forward_rejects_host_or_misshapen_outputs(dev_case):
    _, (q, k, v) = dev_case
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, o=torch.empty((1, 2, 256, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, lse=torch.empty((1, 2, 256), dtype=torch.float32))
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, o=torch.empty((1, 2, 255, 128), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, lse=torch.empty((1, 2, 256), dtype=torch.float16, device="cuda"))
    assert binding.get_device_status() == 0


def test_host_entry_rejects_mismatched_buffers(dev_case):
    case, dev = dev_case
    h = [t.pin_memory() for t in case.stored]
    d_in = [torch.empty_like(t) for t in dev]
    h_o = torch.empty((1, 2, 256, 128), dtype=torch.bfloat16).pin_memory()
    h_l = torch.empty((1, 2, 256), dtype=torch.float32).pin_memory()
    d_o = torch.empty((1, 2, 256, 128), dtype=torch.bfloat16, device="cuda")
    d_l = torch.empty((1, 2, 256), dtype=torch.float32, device="cuda")
    short_o = torch.empty((1, 2, 128, 128), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError):
        binding.attn_fwd_host(*h, short_o, h_l, *d_in, d_o, d_l)
    with pytest.raises(ValueError):  # a device tensor where a host buffer is expected
        binding.attn_fwd_host(dev[0], h[1], h[2], h_o, h_l, *d_in, d_o, d_l)
    with pytest.raises(ValueError):  # a host tensor where a device staging buffer is expected
        binding.attn_fwd_host(*h, h_o, h_l, d_in[0], d_in[1], h[2], d_o, d_l)
    with pytest.raises(ValueError):
        binding.attn_fwd_host(*h, h_o, h_l, *d_in, d_o, d_l[:, :, :100])
    # the same buffers, well formed, go through
    binding.attn_fwd_host(*h, h_o, h_l, *d_in, d_o, d_l)
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0


def test_backward_and_split_reject_host_buffers(dev_case):
    _, (q, k, v) = dev_case
    o, lse = binding.attn_fwd(q, k, v)
    dout = torch.randn_like(q, dtype=torch.float32).to(torch.bfloat16)
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse, dout, dq=torch.empty((1, 2, 256, 128), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse.cpu(), dout)
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, o, lse, dout, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        binding.attn_fwd_split(q, k, v, n_splits=2, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    torch.cuda.synchronize()
    assert binding.get_device_status() == 0
