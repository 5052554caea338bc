"""Attn-QAT (NVFP4 fake-quantized attention) for GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (``libattnqat.so``);
``attnqat`` is its thin ctypes binding and ``synth`` draws seeded inputs.
Importing the package loads nothing; ``attnqat.load()`` opens the library and
fails loudly if it has not been built.
"""
__all__ = ["attnqat", "synth"]
