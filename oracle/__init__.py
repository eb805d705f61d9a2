"""CPU oracle for the ForkAttention token-mixing layer (test infrastructure).

This package is the correctness reference for the CUDA path.  It is *test
infrastructure*: only the tests, the package smoke check and the benchmark's
CPU-baseline leg may import or run it.  It shares no code with the CUDA path
and imports nothing from it.

It computes the plain definition the method reaches exactly (Flide,
"Proposition 3.1" / "Proposition 1": every question's hidden states equal
those of running ``s ⊕ q_i`` on its own): every trunk and every
``s ⊕ q_i`` is run as an independent sequence through the layer definitions
(rotary full / sliding-window attention, short causal conv + gated delta rule,
options softmax).  Arithmetic is float32 by default (the pages compare
engines against a float32 reference) and float64 on request.

Parity status of each function is listed in ``oracle.forkattn.PINS``.
"""
from .forkattn import *  # noqa: F401,F403
