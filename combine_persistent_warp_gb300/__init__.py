"""Fused FP8 Mixture-of-Experts layer ("Mega-MoE") for one GB300 GPU.

The layer is a C-ABI CUDA library (``libcpw_moe.so``, declared in
``include/cpw_moe.h``); :class:`FusedMoE` is a thin ctypes binding over it that uses
PyTorch only for device memory and streams.  ``workloads`` synthesises seeded inputs.
"""
from .native import FusedMoE, MoeError, load  # noqa: F401

__all__ = ["FusedMoE", "MoeError", "load"]
