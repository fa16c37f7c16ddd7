"""GB300-native decode attention for speech-recognition decoders.

The compute lives in ``libasrkv.so`` (hand-written sm_103a CUDA kernels behind
a plain C ABI, declared in include/asrkv.h).  ``kv_cache_decode_asr_gb300.ops``
is a thin ctypes binding with the same names as the C entry points; it only
marshals torch tensors into pointers and sizes.  There is no CPU fallback:
calling an op without the built library raises.
"""
import importlib

__all__ = ["ops", "synthetic"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
