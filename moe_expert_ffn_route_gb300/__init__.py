"""Fused MoE expert FFN forward for one GB300 (sm_103a).

The hot path lives in hand-written CUDA kernels behind the C ABI of
``include/moeffn.h`` (built into ``_build/<machine>/libmoeffn.so`` by
``build.py``); ``binding`` marshals torch tensors to it.  ``synth`` draws the
seeded synthetic workloads.  Nothing is loaded at import time.
"""
__all__ = ["binding", "build", "synth"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
