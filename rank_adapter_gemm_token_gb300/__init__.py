"""GB300 (sm_103a) multi-LoRA batched linear layer.

The compute path is libmlora.so (hand-written CUDA: slot-sort metadata, tcgen05 base GEMM,
shrink/expand side path) behind the C ABI in include/mlora.h; ``mlora`` is its Python
binding and ``layer`` a small convenience wrapper over torch device buffers.
"""
from . import mlora  # noqa: F401

__all__ = ["mlora"]
