"""Slot metadata oracle: sort a step's (token, slot) pairs by slot. TEST INFRASTRUCTURE ONLY.

Source: "Multi-LoRA Serving Explained" (sevydevy.com), the batched-serving demo
("Segmented: sort tokens by adapter, one small matmul per segment"): the
segmented method orders tokens with a *stable* argsort of their slot ids and
groups equal ids; its printed segment counts for the ids [2, 0, -1, 2, 3, 0] are
-1: 1, 0: 2, 2: 2, 3: 1. The same page says the vLLM kernel path sorts the batch's
tokens by slot before shrink and expand.
"[RFC] Per-request activation of multiple LoRA adapters", "Proposed Change" item 2,
generalises the map to k slots per token, unused ones holding the sentinel.

Reading taken here: the k slots of token t are flattened to pair index p = t*k + j,
the pairs are stably sorted by slot value (so -1 comes first and equal slots keep
ascending p), and a segment is a maximal run of equal slot values, listed in
ascending slot order.
"""
from __future__ import annotations


def meta(token_slots, n_slots: int | None = None) -> dict:
    """order (pair indices, stable by slot), seg_slot, seg_off (n_seg + 1 offsets), n_active."""
    flat = [int(v) for row in _rows(token_slots) for v in row]
    if n_slots is not None:
        for v in flat:
            if v != -1 and not 0 <= v < n_slots:
                raise ValueError(f"slot id {v} outside [-1, {n_slots})")
    order = sorted(range(len(flat)), key=lambda p: flat[p])     # Python's sort is stable
    seg_slot, seg_off = [], []
    for i, p in enumerate(order):
        if i == 0 or flat[p] != flat[order[i - 1]]:
            seg_slot.append(flat[p])
            seg_off.append(i)
    seg_off.append(len(order))
    n_active = sum(1 for v in flat if v != -1)
    return dict(order=order, seg_slot=seg_slot, seg_off=seg_off, n_active=n_active)


def _rows(token_slots):
    try:
        import numpy as np
        a = np.asarray(token_slots)
        if a.ndim == 1:
            a = a.reshape(-1, 1)
        return a.tolist()
    except ImportError:  # pragma: no cover
        return [list(r) if isinstance(r, (list, tuple)) else [r] for r in token_slots]
