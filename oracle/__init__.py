"""CPU oracle for the batch-invariant decoder step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import anything in this
package.  The product (``invariant_vd_step_gb300``) never imports it and
shares no code, table or constant with it; the only common module is the
seeded input generator ``invariant_vd_step_gb300.synth``, which draws
inputs and performs none of the decoder's arithmetic.

What it computes.  ``Forward(W, h)`` of Theorem 4.1 in "Vosti: Specifying,
Implementing, and Verifying Deterministic LLM Inference" (深入解析 Vosti,
§二, Theorem 4.1 engine-step preservation): the last-position logits of a
cold causal forward over the token history ``h`` from an empty KV cache, and
``fKV(W, h, p)`` (same page, §五 5.1): the per-layer K/V at position p of
that cold forward.  Batch invariance reaches the mathematically same
result as the plain definition, so the oracle *is* the plain definition,
written out in float64, with no tiling, splitting or reordering:

* every floating-point step is done in float64 on the exact bf16 values;
* results are rounded to bf16 (round-to-nearest-even) at every module
  output (norm, projection, RoPE, attention output, GLU, residual add),
  because the model's dtype (bf16) is part of the configuration W
  (深入解析 Vosti, §二 Definition 2.1: W includes the numeric dtype);
* logits are returned unrounded (float64).

Parity status of each function is stated in its docstring; functions
whose only check is the end-to-end tolerance say "parity unpinned".
"""
