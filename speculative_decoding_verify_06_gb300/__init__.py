"""GB300-native verify pass of speculative decoding for a dense 4-bit-quantised LLM.

The compute lives in ``libsvd.so`` (hand-written CUDA for sm_103a behind the C ABI declared in
``include/svd.h``); :mod:`.svd` is its thin ctypes binding, :mod:`.stack` assembles a whole verify
pass (the 27B-shaped layer stack, lm_head, sampler, acceptance) into one CUDA graph, and
:mod:`.synth` draws the seeded synthetic inputs.  Importing this package loads nothing: the
library is opened on first use and any entry point fails loudly when it is missing.
"""
__all__ = ["svd", "stack", "synth", "roofline", "build"]
