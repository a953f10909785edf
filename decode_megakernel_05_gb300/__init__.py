"""GB300 batch-size-1 decode megakernel: one persistent fused CUDA kernel per token.

``mk`` is the thin binding of the C ABI (``include/mk.h``); ``Decoder`` wraps a
context with torch-allocated device buffers.  All computation runs in the
sm_103a CUDA kernels of ``_build/libmk.so``.
"""
from . import mk
from .decoder import Decoder

__all__ = ["mk", "Decoder"]
