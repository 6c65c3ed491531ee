"""GB300-native (sm_103a) DeepSeek-style Mixture-of-Experts layer forward.

Router (fused gate GEMM + sigmoid + bias + top-k) -> dispatch (histogram, scan, stable
permutation, affinity) -> grouped SwiGLU expert FFN on tcgen05 tensor cores (+ shared
expert) -> combine, behind the C ABI of include/moe.h.  ``binding`` is the thin Python
binding; ``synth`` holds the seeded synthetic input recipes.
"""
import importlib

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
