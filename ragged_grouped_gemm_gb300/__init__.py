"""GB300-native single-GPU dropless MoE layer: a C-ABI library of sm_103a
CUDA kernels (include/moe.h, built into _build/libmoe.so) and its thin
Python binding.

``inputs`` (seeded synthetic workloads) imports without the library; the
binding (``api``) loads libmoe.so on first use and raises if it is missing.
"""
from .inputs import CONFIGS, MoEConfig  # noqa: F401

__all__ = ["CONFIGS", "MoEConfig", "api", "inputs"]


def __getattr__(name):
    if name == "api":
        import importlib
        return importlib.import_module(".api", __name__)
    raise AttributeError(name)
