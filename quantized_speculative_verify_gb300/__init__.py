"""Quantized speculative-verify linear layer for GB300 (sm_103a).

The verify pass of speculative decoding runs the target model over a draft
tree of M tokens; its linear layers rotate the activations with a 32-block
randomized Hadamard transform, quantize them to int8 per row, and multiply
them against 4-bit asymmetric ("Medium") or 8-bit symmetric ("Large")
grouped integer weights that went through the same rotation offline.

The compute lives in libhq.so (C ABI, include/hq.h; CUDA kernels under
csrc/).  ``hq`` is the thin ctypes binding; ``synth`` draws seeded synthetic
inputs.
"""
from . import hq, synth  # noqa: F401

__all__ = ["hq", "synth"]
