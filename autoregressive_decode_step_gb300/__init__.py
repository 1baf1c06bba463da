"""GB300 (sm_103a) single-token decode step for Llama/Qwen-style decoders.

The compute lives in the C-ABI library ``libdecodestep.so`` (hand-written CUDA
kernels, declared in ``include/decode_step.h``).  ``abi`` is its thin ctypes
binding; ``model`` holds the decode driver built on it; ``configs`` and
``synth`` describe the workloads and make their seeded synthetic inputs.

Importing this package loads nothing native; importing ``abi`` does, and fails
loudly when the library has not been built.
"""

__all__ = ["configs", "synth", "abi", "model"]
