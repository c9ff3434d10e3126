"""GB300-native (sm_103a) FlashAttention-2-style attention forward.

The compute lives in a C-ABI shared library of hand-written CUDA kernels
(``tiled_attention_fa2_gb300/_lib/libattn_fa2.so``, declared in
``include/attn_fa2.h``); :mod:`tiled_attention_fa2_gb300.binding` marshals
torch tensors into it.  The binding is imported lazily so that the seeded
input generators (:mod:`tiled_attention_fa2_gb300.inputs`) can be used on a
machine without the library or a GPU.
"""

__all__ = ["attn_fwd", "attn_fwd_fp8", "forward", "inputs"]


def __getattr__(name):
    if name in ("attn_fwd", "attn_fwd_fp8", "forward", "binding"):
        import importlib

        binding = importlib.import_module(__name__ + ".binding")
        return binding if name == "binding" else getattr(binding, name)
    raise AttributeError(name)
