"""GB300-native packed-varlen text-embedding encoder.

The compute lives in a C-ABI CUDA library (``include/tee.h``) built from
``csrc/`` for sm_103a; ``binding`` is its thin ctypes binding and ``synth``
the seeded synthetic-input generator.  Importing the package loads nothing:
``binding.load()`` opens the compiled library and raises if it is missing.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "binding", "build"]
