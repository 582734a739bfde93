"""GB300-native fused attention forward (prefill and split-KV decode).

The compute runs in hand-written sm_103a CUDA kernels inside
``libattn_gb300.so``; :mod:`.binding` marshals torch tensors into the C-ABI
calls declared in ``include/attn.h``.  Importing this package does not load
the library; the first call does, and it raises if the library is missing.
"""
__all__ = ["binding", "inputs"]
