"""fp64 oracle for the multi-LoRA batched linear layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline
leg may import this package; the library (``rank_adapter_gemm_token_gb300``) never does,
and nothing here imports the library. The two share no code.

- ``linear``: the layer's output in fp64 (plain C loops in ``mlora_oracle.c``).
- ``linear_sliced``: a fused linear whose output slices each have their own adapter.
- ``meta``: the per-step slot metadata (stable sort of token/slot pairs by slot).
- ``memory``: the adapter/slot memory arithmetic from the pages.
- ``embedding``: the token embedding lookup with LoRA (``embed.py``, numpy fp64).

Parity pins (tests/test_oracle.py) tie each function to the pages: a hand-worked
example, the merge identity, the PEFT "cat" merge, linearity in the scale, the
sentinel rows, the printed segment counts and the printed memory figures; the sliced
form against the block-diagonal single-adapter identity. The embedding lookup has its own
pins (tests/test_oracle_embedding.py), among them its identity with ``linear`` on one-hot inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import memory  # noqa: F401  (re-export)
from .meta import meta  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mlora_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

ORACLE_OK, ORACLE_ERR_BAD_SLOT, ORACLE_ERR_ARG, ORACLE_ERR_OOM = 0, 1, 2, 3


class OracleError(RuntimeError):
    def __init__(self, code: int):
        names = {ORACLE_ERR_BAD_SLOT: "bad slot id", ORACLE_ERR_ARG: "bad argument",
                 ORACLE_ERR_OOM: "out of memory"}
        super().__init__(f"oracle error {code}: {names.get(code, '?')}")
        self.code = code


def compile_library(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """gcc -O2, no fast-math, no FMA contraction, no -march: the same result on any host."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    return compile_library(force=force)


def _bind(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.oracle_mlora_linear.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                        i32, vp, i32, vp, vp, i32]
    lib.oracle_mlora_linear.restype = i32
    return lib


def load_library(path: str | None = None):
    """Load the compiled oracle (or another build of the same source, for mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def as_f64(a) -> np.ndarray:
    """bf16 bit patterns (uint16) are widened exactly; any float array is cast to float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def linear(x, W, token_slots, adapters, n_slots: int, scales=None, rows=None, cols=None,
           threads: int | None = None, lib=None) -> np.ndarray:
    """y[rows][:, cols] of the multi-LoRA linear in fp64.

    x [T, K], W [D, K]; token_slots [T, J] int (-1 = no adapter); scales [T, J] or None (= 1);
    adapters: mapping slot -> object with A [r, K], B [D, r], rank, alpha, rslora (unpadded).
    """
    x = np.ascontiguousarray(as_f64(x))
    W = np.ascontiguousarray(as_f64(W))
    T, K = x.shape
    D = W.shape[0]
    assert W.shape[1] == K
    ts = np.asarray(token_slots, dtype=np.int32)
    ts = np.ascontiguousarray(ts.reshape(T, ts.shape[-1] if ts.ndim == 2 else 1))
    J = ts.shape[1]
    sc = None if scales is None else np.ascontiguousarray(np.asarray(scales, dtype=np.float64).reshape(T, J))
    keep = []
    A_ptr = (ctypes.c_void_p * max(n_slots, 1))()
    B_ptr = (ctypes.c_void_p * max(n_slots, 1))()
    rank = np.zeros(max(n_slots, 1), dtype=np.int32)
    alpha = np.zeros(max(n_slots, 1), dtype=np.float64)
    rs = np.zeros(max(n_slots, 1), dtype=np.int32)
    for s, ad in (adapters or {}).items():
        if ad is None:
            continue
        assert 0 <= s < n_slots
        A = np.ascontiguousarray(as_f64(ad.A))
        B = np.ascontiguousarray(as_f64(ad.B))
        assert A.shape == (ad.rank, K) and B.shape == (D, ad.rank), (A.shape, B.shape)
        keep += [A, B]
        A_ptr[s] = A.ctypes.data
        B_ptr[s] = B.ctypes.data
        rank[s], alpha[s], rs[s] = ad.rank, ad.alpha, int(bool(ad.rslora))
    r_idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    c_idx = None if cols is None else np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
    n_rows = T if r_idx is None else len(r_idx)
    n_cols = D if c_idx is None else len(c_idx)
    y = np.zeros((n_rows, n_cols), dtype=np.float64)
    lib = lib or load_library()
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    rc = lib.oracle_mlora_linear(T, K, D, J, ptr(x), ptr(W), ptr(ts), ptr(sc), n_slots, A_ptr, B_ptr,
                                 ptr(rank), ptr(alpha), ptr(rs), n_rows, ptr(r_idx), n_cols, ptr(c_idx),
                                 ptr(y), threads or default_threads())
    if rc != ORACLE_OK:
        raise OracleError(rc)
    return y


def linear_sliced(x, W, token_slots, adapters, n_slots: int, widths, scales=None, rows=None,
                  threads: int | None = None) -> np.ndarray:
    """A fused linear (merged qkv / gate_up) whose D = sum(widths) outputs are consecutive slices,
    each with its own adapter ("LoRA Serving" (vLLM learning book, ch. 09-04), section 7: the merged
    column linear applies each sub-projection's adapter separately). adapters: slot -> list with one
    adapter object per slice (A [r, K], B [widths[i], r], rank, alpha, rslora). Each slice is
    computed as its own linear: W rows of the slice with that slice's adapters."""
    W = np.asarray(W)
    out, off = [], 0
    for i, w in enumerate(widths):
        ad_i = {s: a[i] for s, a in (adapters or {}).items()}
        out.append(linear(x, W[off:off + w], token_slots, ad_i, n_slots, scales=scales, rows=rows,
                          threads=threads))
        off += w
    assert off == W.shape[0]
    return np.concatenate(out, axis=1)


from .embed import embedding  # noqa: E402,F401  (re-export; needs OracleError above)
