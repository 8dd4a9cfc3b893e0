"""GB300-native k-quant MMQ prefill GEMM: Y[T x O] = X[T x K] . W[O x K]^T
with W in q4_K or q6_K and X quantised per 32-element block to q8_1.

The compute path is the C-ABI library ``libmmq.so`` (hand-written sm_103a
CUDA); :mod:`.ops` is the thin Python binding over it.  Importing this
package does not load the library; the first op call does, and raises if
the library or a GPU is missing.
"""
import importlib

__all__ = ["ops", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
