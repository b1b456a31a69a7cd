"""CPU float64 oracle for exact softmax attention (test infrastructure).

This package is test infrastructure, not part of the product. Only the test
suite, the smoke check and the CPU-baseline leg of the benchmark may import
or run it. It shares no code, header, table or helper with the CUDA path,
and the CUDA path never imports it.

Modules
-------
attention
    The plain definition: softmax(scale * Q K^T) V with the mask applied,
    log-sum-exp per row, and the closed-form gradients, all in float64 with
    the full score row of each query materialised.
tiled
    The tiled restatement with an online softmax (one key block at a time),
    used only to check the block-size invariance the pages promise.

Every function is pinned by a CPU test against something other than itself:
the worked examples printed on "Tiled attention with an online softmax"
(section "Examples"), closed forms, brute-force scalar loops on tiny inputs,
central finite differences, and CPU float64 ``torch.autograd``.
"""
from . import attention, tiled  # noqa: F401

__all__ = ["attention", "tiled"]
