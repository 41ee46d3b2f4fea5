"""GB300-native MXFP4 lightning-indexer path.

The compute lives in ``libidx.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/idx.h``); ``binding`` marshals PyTorch tensors to it.
``workloads`` draws seeded synthetic inputs and needs no GPU.
"""
from . import workloads  # noqa: F401


def __getattr__(name):
    # The binding loads the CUDA library; import it only when an op is used so
    # that the CPU-only parts of the package import without it.
    from . import binding
    return getattr(binding, name)
