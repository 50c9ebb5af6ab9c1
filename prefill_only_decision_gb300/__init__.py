"""Prefill-only decisions on a hybrid (gated delta-rule + GQA) decoder for GB300 (sm_103a).

The compute path lives in the CUDA library `libs1.so` built from `csrc/`; the
Python side is a ctypes binding (`binding`). Importing this package does not
load the library; `binding.lib()` does, and fails loudly when it is missing.
"""
__all__ = ["configs", "synth", "binding"]
