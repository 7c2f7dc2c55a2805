"""Adapter memory arithmetic. TEST INFRASTRUCTURE ONLY.

Source: "Multi-LoRA Serving Explained" (sevydevy.com), the memory-maths section and
the max-lora-rank section. An adapted layer stores rank * (input + output) numbers
(A is rank x input, B is output x rank); a model's adapter multiplies that over its
layers and by bytes per number; a GPU slot is reserved at the maximum rank. The
page's made-up model: 32 blocks of seven linears (q, k, v, o at hidden 4096 with k
and v emitting 1024; gate and up widening to 14336; down narrowing back), 16-bit
numbers, plus input and output embeddings of 100,000 x 4096.
"""
from __future__ import annotations

LAYERS, HIDDEN, KV_OUT, MLP, VOCAB, BYTES = 32, 4096, 1024, 14336, 100_000, 2

# (input width, output width) of each adapted linear of one block
MODULES = {
    "q": (HIDDEN, HIDDEN), "k": (HIDDEN, KV_OUT), "v": (HIDDEN, KV_OUT), "o": (HIDDEN, HIDDEN),
    "gate": (HIDDEN, MLP), "up": (HIDDEN, MLP), "down": (MLP, HIDDEN),
}


def base_bytes() -> int:
    weights = LAYERS * sum(i * o for i, o in MODULES.values())
    return (weights + 2 * VOCAB * HIDDEN) * BYTES


def adapter_bytes(rank: int) -> int:
    return LAYERS * sum(rank * (i + o) for i, o in MODULES.values()) * BYTES


def slot_bytes(n_slots: int, max_rank: int) -> int:
    return n_slots * adapter_bytes(max_rank)
