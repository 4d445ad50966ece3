"""GB300-native paged BF16 operators (PSI hot path): C-ABI library libpsi
(tcgen05/TMA CUDA kernels for sm_103a) plus a ctypes binding.

``psi``       the binding: one Python function per C entry point
``torch_io``  device/pinned memory and streams from PyTorch
``build``     in-tree nvcc build of libpsi.so
"""
from . import psi  # noqa: F401

__all__ = ["psi"]
