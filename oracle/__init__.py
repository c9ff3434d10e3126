"""Float64 CPU oracle for the FlashAttention-2-style attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product path (the CUDA library and its Python binding) never imports, calls or
links anything here, and nothing here imports the product package.

Sources the oracle follows (page title, then the section or listing cited):

* "Kernels and Memory in LLM Inference", section "Attention, said plainly again"
  -- the definition: scores S = Q K^T, a row softmax with the row max subtracted,
  then a weighted sum of V; heads are independent.
* "FlashAttention-2 from PyTorch to Triton" -- the opening description of the FA2
  forward pass (running m, l, unnormalised O, one division by l at the end, and
  L = m + log l), its PyTorch double-loop listing, its causal convention
  (key j kept iff j <= query i) and its test reference (SDPA plus a logsumexp of
  the masked scaled scores).
* "1.8x Faster Attention on an RTX 5080: an FP8 Flash Attention Kernel in
  CuTe-DSL", sections "The attention itself" (online softmax worked example) and
  "Who am I, what's mine?" (FP8 descales folded into the score scale).
* Grouped-query attention ("Kernels and Memory in LLM Inference", "Store less:
  MQA, GQA, MLA", "Grouped-query attention (2023)"): groups of query heads share
  one K/V head; each query head is ordinary attention against its group's head.
* The backward pass ("FlashAttention-2 from PyTorch to Triton", item 5 of the
  list of what its first kernel leaves out; "Kernels and Memory in LLM
  Inference", "Training detour (brief)"): P rebuilt from L, D = rowsum(dO * O),
  dK and dV per key tile, dQ accumulated; the gradient formulas are the chain
  rule on the forward's definition.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
worked values printed on those pages, closed forms, invariants and a
high-precision brute force; none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    e4m3_bits_to_f64,
    dequantize,
    attention_probs,
    attention_reference,
    attention_rows,
    attention_tiled,
    kv_head_of,
    attention_gqa,
    attention_gqa_rows,
    attention_backward,
    attention_backward_tiled,
)
