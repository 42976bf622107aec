"""GB300 (sm_103a) W8A8 MXFP8 linear layer.

The compute runs in the CUDA library ``libmxfp8.so`` built from ``csrc/``; the
Python module :mod:`.ops` is a thin ctypes binding over its C ABI.  Importing
this package does not load the library; the first call into :mod:`.ops` does,
and raises if it is missing or no sm_103 GPU is present.
"""

__all__ = ["ops", "synth"]
