"""Rotation-quantized (RotorQuant PlanarQuant / IsoQuant) KV cache for GB300 (sm_103a).

`rq` is the binding of the C-ABI library librq.so (include/rq.h); `synth` draws the seeded
synthetic workloads.  Importing the package loads nothing; the library is built and loaded on
first use.
"""
__all__ = ["rq", "synth"]
