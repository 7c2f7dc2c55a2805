"""Torch-facing convenience objects over the C ABI (argument marshalling only).

``AdapterPool`` owns one adapted linear's slot pool, ``StepMeta`` one step's slot
metadata, and ``linear`` runs the layer y = x W^T + sum_j s c B(A x) into an fp32 tensor.
Torch provides device memory and streams; every step of the computation runs in
libmlora.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import mlora


def bf16_from_bits(bits: np.ndarray, device=None) -> torch.Tensor:
    """A bf16 tensor holding the given 16-bit patterns (numpy uint16)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def _pinned_bits(a) -> torch.Tensor:
    if isinstance(a, torch.Tensor):
        t = a.detach().contiguous().cpu().view(torch.int16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.pin_memory() if torch.cuda.is_available() else t


class AdapterPool:
    """The slots of one adapted linear: A [C, K] and B [D, C] (bf16, zero padded) over a column
    space in which slot s owns its rank rows. With `classes` = [(n_slots_c, rank_c), ...] the slots
    come in rank classes (numbered class by class); otherwise n_slots slots of rank r_max."""

    def __init__(self, n_slots: int, r_max: int, K: int, D: int, copy_stream=None, classes=None):
        self.K, self.D = K, D
        if classes:
            self.classes = [(int(n), int(r)) for n, r in classes]
            self.n_slots = sum(n for n, _ in self.classes)
            self.r_max = max(r for _, r in self.classes)
            self.handle = mlora.mlora_pool_create_classes([n for n, _ in self.classes], [r for _, r in self.classes],
                                                          K, D, copy_stream)
        else:
            self.classes = None
            self.n_slots, self.r_max = n_slots, r_max
            self.handle = mlora.mlora_pool_create(n_slots, r_max, K, D, copy_stream)
        self._staged = []           # pinned host copies kept alive until the next sync

    def load(self, slot: int, A, B, rank: int, alpha: float, rslora: bool = False) -> None:
        a, b = _pinned_bits(A), _pinned_bits(B)
        assert a.numel() == rank * self.K and b.numel() == self.D * rank
        self._staged += [a, b]
        mlora.mlora_load_adapter(self.handle, slot, a.data_ptr(), b.data_ptr(), rank, alpha, rslora)

    def clear(self, slot: int) -> None:
        mlora.mlora_clear_slot(self.handle, slot)

    def sync(self) -> None:
        mlora.mlora_pool_sync(self.handle)
        self._staged.clear()

    def info(self) -> dict:
        return mlora.mlora_pool_info(self.handle)

    def layout(self) -> dict:
        return mlora.mlora_pool_layout(self.handle, self.n_slots)

    def close(self) -> None:
        if self.handle:
            mlora.mlora_pool_destroy(self.handle)
            self.handle = 0
            self._staged.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class EmbeddingPool(AdapterPool):
    """The slots of an embedding table with LoRA: A kept token-major ([vocab, C]), B [dim, C].
    load() takes each adapter's A [rank, vocab] and B [dim, rank], like a linear pool with
    K = vocab and D = dim."""

    def __init__(self, vocab: int, dim: int, classes, copy_stream=None):
        self.K, self.D = vocab, dim
        self.classes = [(int(n), int(r)) for n, r in classes]
        self.n_slots = sum(n for n, _ in self.classes)
        self.r_max = max(r for _, r in self.classes)
        self.handle = mlora.mlora_embedding_pool_create([n for n, _ in self.classes], [r for _, r in self.classes],
                                                        vocab, dim, copy_stream)
        self._staged = []


class StepMeta:
    """Per-step slot metadata for up to max_tokens tokens with J slots each."""

    def __init__(self, max_tokens: int, J: int, r_max: int):
        self.max_tokens, self.J_max, self.r_max = max_tokens, J, r_max
        self.handle = mlora.mlora_meta_create(max_tokens, J, r_max)
        self.T = 0
        self.J = J

    def build(self, token_slots: torch.Tensor, scales: torch.Tensor | None, pool: AdapterPool, stream=None) -> None:
        assert token_slots.is_cuda and token_slots.dtype == torch.int32 and token_slots.is_contiguous()
        T, J = (token_slots.shape[0], token_slots.shape[1]) if token_slots.dim() == 2 else (token_slots.shape[0], 1)
        if scales is not None:
            assert scales.is_cuda and scales.dtype == torch.float32 and scales.numel() == T * J
        mlora.mlora_build_meta(self.handle, token_slots, scales, T, J, pool.handle, _stream(stream))
        self.T, self.J = T, J

    def status(self) -> None:
        mlora.mlora_meta_status(self.handle)

    def read(self) -> dict:
        return mlora.mlora_meta_read(self.handle, self.T * self.J)

    def close(self) -> None:
        if self.handle:
            mlora.mlora_meta_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream()
    return stream


def linear(pool: AdapterPool, meta: StepMeta, x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """y[T, D] fp32 = x W^T + the step's LoRA side path (x [T, K] and W [D, K] bf16 on the GPU)."""
    assert x.dtype == torch.bfloat16 and W.dtype == torch.bfloat16 and x.is_contiguous() and W.is_contiguous()
    T = meta.T
    assert x.shape == (T, pool.K) and W.shape == (pool.D, pool.K)
    if y is None:
        y = torch.empty((T, pool.D), dtype=torch.float32, device=x.device)
    mlora.mlora_linear(pool.handle, meta.handle, x, W, y, _stream(stream))
    return y


def embedding(pool: EmbeddingPool, meta: StepMeta, ids: torch.Tensor, E: torch.Tensor, y: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """y[T, dim] fp32 = E[ids] + the step's LoRA side path (ids int32 [T], E [vocab, dim] bf16 on the GPU)."""
    assert ids.dtype == torch.int32 and E.dtype == torch.bfloat16 and ids.is_contiguous() and E.is_contiguous()
    T = meta.T
    assert ids.shape == (T,) and E.shape == (pool.K, pool.D)
    if y is None:
        y = torch.empty((T, pool.D), dtype=torch.float32, device=E.device)
    mlora.mlora_embedding(pool.handle, meta.handle, ids, E, y, _stream(stream))
    return y


def base_gemm(x: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    T, K = x.shape
    D = W.shape[0]
    if y is None:
        y = torch.empty((T, D), dtype=torch.float32, device=x.device)
    mlora.mlora_base_gemm(x, W, y, T, K, D, _stream(stream))
    return y
