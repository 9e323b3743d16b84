"""Chunkwise gated delta rule (GDN / KDA) forward pass for GB300 (sm_103a).

The compute lives in ``libgdn.so`` (CUDA, C ABI declared in ``include/gdn.h``);
:mod:`.gdn` is a thin ctypes binding with the same names, and :mod:`.synth`
draws seeded synthetic inputs.  There is no CPU fallback: calling the op
without the compiled library raises.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "gdn"]


def __getattr__(name):
    if name == "gdn":
        from . import gdn as _gdn
        return _gdn
    raise AttributeError(name)
