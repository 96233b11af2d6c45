"""GB300-native exact tiled attention forward (sm_103a).

The compute path is the C-ABI library ``libfa.so`` built from ``csrc/``;
``api`` only marshals arguments into it. ``workloads`` holds the seeded
synthetic input generators and nothing of the method; ``accounting`` the
FLOP / byte conventions used for measurement.
"""
from . import accounting, api, workloads  # noqa: F401

__all__ = ["accounting", "api", "workloads"]
