"""SpeContext decode-step hot path for GB300 (sm_103a).

The compute path is the C-ABI library ``libspc.so`` (CUDA kernels, declared in
``include/spc.h``); ``binding`` marshals arguments to it and ``pipeline`` runs
a decode step on two CUDA streams. The library is loaded on first use and a
missing or unloadable library raises; there is no CPU fallback.
"""
from .configs import CONFIGS, Workload, scaled, describe  # noqa: F401

__all__ = ["CONFIGS", "Workload", "scaled", "describe"]
