"""GVA (Grouped Value Attention) decode hot path for NVIDIA B300 (sm_103a).

The compute lives in libgva.so (C ABI, include/gva.h), built by
`python -m compact_kv_cache_gva_b300.build`.  `gva` is the thin ctypes binding with the C
names, `layer.GVADecodeLayer` runs one decode step, `synth` draws seeded inputs.
"""
__all__ = ["gva", "layer", "synth"]
