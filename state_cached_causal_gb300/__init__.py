"""State-cached causal short convolution on GB300 (sm_103a).

The compute path is ``libcconv.so`` (hand-written CUDA, C ABI, declared in
``include/cconv.h``); ``state_cached_causal_gb300.ops`` is the thin ctypes
binding with the same entry-point names. Importing this package does not load
the library: ``ops`` loads it on first use and raises if it is missing.
"""
import importlib

__all__ = ["ops", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
