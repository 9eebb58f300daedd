"""VC-Attention hot path for GB300 (sm_103a): V-Smooth + ExpCast-FP8 attention.

The compute lives in ``libvca.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/vca.h``).  ``bit_attention_video_smooth_gb300.vca`` is the
thin ctypes binding with the same entry-point names; it is imported lazily so
that the seeded input generator (``inputs``) can be used without the library.
"""
import importlib

__all__ = ["vca", "inputs"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
