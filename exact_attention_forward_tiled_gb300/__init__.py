"""GB300-native exact tiled attention forward (sm_103a).

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``; the
Python names below only marshal arguments into it (``api``). ``workloads``
holds the seeded synthetic input generators and nothing of the method.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "api"]


def __getattr__(name):
    if name == "api":
        from . import api
        return api
    raise AttributeError(name)
