"""Bitwise-deterministic MoE grouped GEMM with a private-slot dprob epilogue,
for GB300 (sm_103a).

The compute path lives in ``libdmoe.so`` (hand-written CUDA behind a C ABI,
declared in ``include/dmoe.h``); ``api`` is a thin ctypes binding that passes
torch tensors' device pointers and the current stream.  Importing this package
does not load the library; the first call into ``api`` does, and fails loudly
if it has not been built.
"""
import importlib

__all__ = ["api", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
