"""B300-native MoE layer hot path: route -> dispatch -> expert FFN -> combine.

The compute lives in a C-ABI CUDA library (``libmoe.so``, declared in
``include/moe.h``); ``expert_routing_router_b300.moe`` is its thin ctypes binding.
``workloads`` draws the seeded synthetic inputs.  The binding is imported lazily
so that input generation works on machines without the built library.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "moe"]


def __getattr__(name):
    if name == "moe":
        import importlib
        return importlib.import_module(__name__ + ".moe")
    raise AttributeError(name)
