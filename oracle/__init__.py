"""Oracle: a plain, slow, CPU implementation of the prefill-only decision path.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports, links or runs this
package; only the tests, the smoke check and the benchmark's CPU-baseline leg
do. It shares no code with the CUDA path: both receive the same arrays from
the seeded input generator and compute independently.

Modules
  gdn      gated delta rule: token recurrence and the chunked (WY) form
  model    RMSNorm, LoRA linear, RoPE, attention, SwiGLU, the hybrid decoder
           forward (unbranched and prefix-branched) and the decision readout

Precision: float32 by default (the pages compare against a float32
reference: System1-Omni issue #10, the mistral.rs worker's parity note, and
the sys1rust README's "upstream PyTorch fp32 reference"); every function
takes a dtype so the self-tests can run it in float64.

Parity status: every function is pinned by a test in tests/test_oracle_*.py
against closed forms, special cases, library routines or brute force. The
end-to-end decision values on random weights have no published worked
example ("parity unpinned" for the composed numbers); they are pinned only
through their parts and invariants.
"""
