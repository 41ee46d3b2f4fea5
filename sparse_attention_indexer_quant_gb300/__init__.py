"""GB300-native MXFP4 lightning-indexer path.

The compute lives in ``libidx.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/idx.h``); ``binding`` marshals PyTorch tensors to it.
``workloads`` draws seeded synthetic inputs and needs no GPU.
"""
import importlib

_SUBMODULES = {"binding", "build_lib", "workloads"}


def __getattr__(name):
    # The binding loads the CUDA library; it is imported only when an op is
    # used, so that the CPU-only parts of the package import without it.
    if name in _SUBMODULES:
        return importlib.import_module(f".{name}", __name__)
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(importlib.import_module(".binding", __name__), name)
