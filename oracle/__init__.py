"""Plain, slow, CPU reference ("oracle") for the River-LLM KV-shared exit river.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only the test-suite, the smoke check and the
benchmark's CPU-baseline leg do.  It shares no code with the CUDA library and
imports nothing from it; both take their inputs from the seeded generators in
``synth``.

Precision: fp32 (NumPy), as the method's specification fixes ("a plain fp32
CPU transformer").  The quantizer follows IEEE fp32 / fp16 rounding exactly,
since its integer output must match the library bit for bit.

Source of the method: the River-LLM explainer page ("River-LLM: Large
Language Model Seamless Exit Based on KV Share"), sections 三 (exit layers:
parameter copies shrunk to W4A16, sharing the backbone's KV cache), 四 (exit
decision: state-transition similarity, minimum over the parallel tokens,
compared with tau, monotone in depth) and 五 (sequence-level exit in prefill,
token-level exit in generation).

Pins: every function here is checked against something other than itself in
``tests/test_oracle_*.py`` (closed forms, library routines, brute force,
invariants of the method).  No function is "parity unpinned".
"""
from .quant import quantize_linear, dequantize_linear, unpack_nibbles
from .model import OracleModel, Policy, rmsnorm, rope, attention, silu, cosine

__all__ = [
    "quantize_linear", "dequantize_linear", "unpack_nibbles",
    "OracleModel", "Policy", "rmsnorm", "rope", "attention", "silu", "cosine",
]
