"""fp64 oracle for LoRA on the token embedding lookup.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the tests, the smoke check and the
benchmark's CPU-baseline leg may call it; the library never does.

What it computes. "[vLLM] LoRA" (secrett2633 blog), layer-implementation section, lists an
embedding variant of the LoRA layers (VocabParallelEmbeddingWithLoRA), and "LoRA Serving" (vLLM
learning book ch. 09-04), section 2, places it beside the linear variants, all served through the
same per-token slot mapping (sections 4.2 and 6). Neither page writes its arithmetic out; the
plainest reading that the rest supports is the LoRA definition itself applied to the lookup:

    an embedding table E [V, D] maps token id i to the row E[i], which is the linear map
    x -> x E applied to the one-hot vector x = e_i. A LoRA adapter of that map has A [r, V] and
    B [D, r] ("Multi-LoRA Serving Explained", LoRA basics: B is d x r, A is r x k, with k the
    input width, here the vocabulary) and adds c B (A e_i) = c B A[:, i], c = alpha / r
    (alpha / sqrt(r) under rsLoRA, "[vLLM] LoRA", PEFTHelper).

With k slots per token and per-(token, slot) scales ("[RFC] Per-request activation of multiple
LoRA adapters", Proposed Change), one token t with id i receives

    y[t] = E[i] + sum_{j : slot[t, j] != -1} s[t, j] c(slot) B_slot A_slot[:, i].

So the shrink of the linear layer becomes a gather of one column of A, and the expand is the
linear layer's expand. Steps follow that order: the token's row of the table, then per slot the
column of A, its product with B (a library matrix-vector product), scaled and added.

Pins (tests/test_oracle_embedding.py): the one-hot identity against the linear-layer oracle (the
C loops of mlora_oracle.c, not this code), a hand-worked example with plain and rsLoRA adapters
(tests/golden/embedding_hand.txt), sentinel rows equal to the table's row bit for bit, the merged
table E + c (B A)^T, and planted mistakes that the pins must catch.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    """bf16 bit patterns (uint16) widened exactly; any other array cast to float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def embedding(ids, E, token_slots, adapters, n_slots: int, scales=None, rows=None) -> np.ndarray:
    """y[rows] of the embedding lookup with LoRA, in fp64.

    ids [T] token ids in [0, V); E [V, D] (bf16 bits or floats); token_slots [T, J] (-1 = no
    adapter); scales [T, J] or None (= 1); adapters: slot -> object with A [r, V], B [D, r],
    rank, alpha, rslora. rows: token indices to compute (default all). A token id outside
    [0, V), a slot outside [-1, n_slots) or a slot with no adapter raises ValueError."""
    from . import ORACLE_ERR_ARG, ORACLE_ERR_BAD_SLOT, OracleError

    E = np.asarray(E)
    V, D = E.shape
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    T = ids.shape[0]
    ts = np.asarray(token_slots, dtype=np.int64).reshape(T, -1) if T else np.zeros((0, 1), np.int64)
    J = ts.shape[1]
    sc = None if scales is None else np.asarray(scales, dtype=np.float64).reshape(T, J)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    adapters = adapters or {}
    B64 = {}                                   # slot -> B in float64, converted once
    y = np.zeros((len(rows), D), dtype=np.float64)
    for n, t in enumerate(rows):
        i = int(ids[t])
        if not 0 <= i < V:
            raise OracleError(ORACLE_ERR_ARG)
        acc = _f64(E[i]).copy()                # the token's row of the table
        for j in range(J):
            s = int(ts[t, j])
            if s == -1:
                continue
            ad = adapters.get(s) if 0 <= s < n_slots else None
            if ad is None:
                raise OracleError(ORACLE_ERR_BAD_SLOT)
            A = np.asarray(ad.A)
            assert A.shape == (ad.rank, V), (A.shape, ad.rank, V)
            if s not in B64:
                B64[s] = _f64(ad.B)
                assert B64[s].shape == (D, ad.rank), (B64[s].shape, D, ad.rank)
            c = float(ad.alpha) / (np.sqrt(float(ad.rank)) if ad.rslora else float(ad.rank))
            a_col = _f64(A[:, i])              # A e_i: the token's column of A
            side = B64[s] @ a_col              # B (A e_i)
            acc += (1.0 if sc is None else float(sc[t, j])) * c * side
        y[n] = acc
    return y
