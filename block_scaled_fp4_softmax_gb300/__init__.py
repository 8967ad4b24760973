"""GB300 (sm_103a) routed mixture-of-experts FFN with block-scaled FP4 experts.

The computation lives in a C-ABI CUDA library (``include/moe.h``, sources in
``csrc/``); :mod:`.moe` is its ctypes binding and :mod:`.synth` the seeded
synthetic input generators.  Importing the package loads nothing; the library
is loaded on first use and must have been built (:func:`.build.build`).
"""

__all__ = ["build", "moe", "synth"]
