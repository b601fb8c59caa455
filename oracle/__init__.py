"""CPU fp64 oracle for the attention forward/backward (test infrastructure).

This package is test infrastructure. Only the test suite, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import it. The product path (the CUDA library and its Python
binding) never calls it, and it shares no code with the product path.

Sources (web pages, cited by title and section):
  * "解析 FlashAttention（3）：FlashAttention-v1 反向传播" (FlashAttention-v1
    backward derivation), §1.1, §2.2-2.7 (eq. 1-8), §3.2 (eq. 9).
  * "反向传播算法详解" (Inference Cookbook, backward pass in detail),
    §1.2-1.3, §2.1 (1)-(5) including the softcap derivative, §8.5 (GQA).
  * Dropout: "解析 FlashAttention（3）" §3.3 and Algorithm 4 of §4; the keep
    mask comes from Philox4x32-10 (Salmon et al., SC 2011), written out in
    ``oracle/philox.py`` from its published definition.

Every function here is pinned by ``tests/test_oracle_pins.py`` (hand-derived
N=2, d=2 example, finite differences against an independent scalar forward,
invariants and special cases).
"""
from .attention import (  # noqa: F401
    attention_forward,
    attention_backward,
    head_forward,
    head_backward,
)
from .philox import dropout_keep_mask, keep_threshold, philox4x32_10  # noqa: F401
