"""Single-GPU MoE layout / dispatch / combine for GB300 (sm_103a).

The expert-parallel ranks are logical destination partitions in one GPU's
HBM. ``binding`` exposes the C ABI of ``libmoe_get.so`` (hand-written CUDA
kernels) on torch tensors; ``workloads`` draws the seeded synthetic inputs.
``binding`` is imported on first use so that building or loading the CUDA
library happens only when it is needed.
"""
import importlib

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
