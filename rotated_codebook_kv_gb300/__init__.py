"""Rotated-codebook KV-cache compression and compressed-KV decode attention (sm_103a).

The compute path is the C-ABI library ``libtq.so`` (``include/tq.h``), built
in-tree from ``csrc/``; ``native`` binds it with ctypes and ``Codec`` marshals
torch tensors into its calls.  ``workloads`` draws seeded synthetic inputs.
"""
from .codec import Codec  # noqa: F401

__all__ = ["Codec"]
