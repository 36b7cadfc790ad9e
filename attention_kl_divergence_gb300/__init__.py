"""libstreamkl: the fused attention KL divergence (StreamKL) on one GB300.

The compute path is the C-ABI library built from ``csrc/`` for sm_103a;
``streamkl`` is its Python binding.  Importing this package does not load the
library; the first call does, and fails loudly if it is missing.
"""
from .inputs import WORKLOADS, Workload, make_g, make_qk, make_workload  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_g", "make_qk", "make_workload", "streamkl"]


def __getattr__(name):
    if name == "streamkl":
        import importlib
        return importlib.import_module(__name__ + ".streamkl")
    raise AttributeError(name)
