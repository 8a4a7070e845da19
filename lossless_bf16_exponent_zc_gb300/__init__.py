"""Lossless BF16 exponent coding (ZipCCL-style) on GB300: a C-ABI CUDA library and its Python binding."""
from . import zc  # noqa: F401

__all__ = ["zc"]
