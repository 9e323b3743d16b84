"""Chunkwise gated delta rule (GDN / KDA) forward pass for GB300 (sm_103a).

The compute lives in ``libgdn.so`` (CUDA, C ABI declared in ``include/gdn.h``);
``chunkwise_gated_delta_gdn_gb300.gdn`` is a thin ctypes binding with the same
names, and :mod:`.synth` draws seeded synthetic inputs.  There is no CPU
fallback: calling the op without the compiled library raises.
"""
