"""Single-GPU (B300, sm_103a) forward pass of one sparse Mixture-of-Experts layer.

The compute lives in the C-ABI library ``libmoe.so`` (``csrc/``); the
functions exported here are the thin ctypes binding to it (see ``binding``).
"""
from .configs import CONFIGS, MoEConfig  # noqa: F401
