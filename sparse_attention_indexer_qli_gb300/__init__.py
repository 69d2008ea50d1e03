"""GB300-native quantized lightning indexer (QLI).

The indexer runs in the C-ABI library ``libqli_gb300.so`` (hand-written
sm_103a CUDA kernels); :mod:`.qli` is its thin Python binding and
:mod:`.synth` the seeded input generator. Importing the package loads nothing
native; the first call into :mod:`.qli` does, and fails loudly when the
library or a CUDA device is missing.
"""
from . import qli, synth  # noqa: F401

__all__ = ["qli", "synth"]
