"""Python binding of mlora.h: argument marshalling only.

Every function below calls the entry point of the same name in libmlora.so; all compute
runs in that library's CUDA kernels. Device buffers are passed as torch tensors (or raw
integer addresses), streams as torch.cuda.Stream (or raw handles). The library must have
been built (``rank_adapter_gemm_token_gb300.build.build()``); if it is missing this module
raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MLORA_OK = 0
MLORA_ERR_INVALID_ARG = 1
MLORA_ERR_SLOT_RANGE = 2
MLORA_ERR_RANK_TOO_LARGE = 3
MLORA_ERR_RANK_INVALID = 4
MLORA_ERR_BAD_TOKEN_SLOT = 5
MLORA_ERR_TOO_MANY_TOKENS = 6
MLORA_ERR_OOM = 7
MLORA_ERR_CUDA = 8
MLORA_ERR_DEVICE_TIMEOUT = 9
MLORA_ERR_MISMATCH = 10
MLORA_ERR_NO_FREE_SLOT = 11
MLORA_ERR_BAD_TOKEN_ID = 12

KERNEL_KINDS = ("meta", "base_gemm", "shrink", "expand", "slot", "embedding")

EXPORTS = (
    "mlora_pool_create", "mlora_pool_destroy", "mlora_load_adapter", "mlora_clear_slot", "mlora_pool_sync",
    "mlora_pool_info", "mlora_pool_bytes", "mlora_meta_create", "mlora_meta_destroy", "mlora_build_meta",
    "mlora_meta_status", "mlora_meta_read", "mlora_linear", "mlora_base_gemm", "mlora_lora_shrink",
    "mlora_lora_expand", "mlora_status_string", "mlora_last_error", "mlora_version", "mlora_launch_count",
    "mlora_trace_enable", "mlora_trace_disable", "mlora_trace_read", "mlora_kernel_kind_name",
    "mlora_lora_apply_noalloc", "mlora_set_gemm_tile_n", "mlora_set_skinny_form", "mlora_check_wait_timeout",
    "mlora_load_adapter_sliced", "mlora_slot_cache_create", "mlora_slot_cache_destroy", "mlora_slot_cache_assign",
    "mlora_slot_cache_lookup", "mlora_slot_cache_pin", "mlora_slot_cache_evict", "mlora_adapter_cache_create",
    "mlora_adapter_cache_destroy", "mlora_adapter_cache_register", "mlora_adapter_cache_unregister",
    "mlora_adapter_cache_pin", "mlora_adapter_cache_map", "mlora_pool_create_classes", "mlora_pool_layout",
    "mlora_set_path", "mlora_embedding_pool_create", "mlora_embedding",
)


class MloraError(RuntimeError):
    def __init__(self, status: int, fn: str, message: str):
        super().__init__(f"{fn}: status {status} ({message})")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libmlora.so (raises FileNotFoundError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise FileNotFoundError(f"{p} is missing: build it with rank_adapter_gemm_token_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, f32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
        sig = {
            "mlora_pool_create": [i32, i32, i32, i32, vp, vp],
            "mlora_pool_create_classes": [i32, vp, vp, i32, i32, vp, vp],
            "mlora_pool_layout": [vp, vp, vp, vp],
            "mlora_set_path": [i32],
            "mlora_embedding_pool_create": [i32, vp, vp, i32, i32, vp, vp],
            "mlora_embedding": [vp, vp, vp, vp, vp, vp],
            "mlora_pool_destroy": [vp],
            "mlora_load_adapter": [vp, i32, vp, vp, i32, f32, i32],
            "mlora_clear_slot": [vp, i32],
            "mlora_pool_sync": [vp],
            "mlora_pool_info": [vp, vp, vp, vp, vp, vp, vp, vp, vp],
            "mlora_meta_create": [i32, i32, i32, vp],
            "mlora_meta_destroy": [vp],
            "mlora_build_meta": [vp, vp, vp, i32, i32, vp, vp],
            "mlora_meta_status": [vp],
            "mlora_meta_read": [vp, vp, vp, vp, vp, vp],
            "mlora_linear": [vp, vp, vp, vp, vp, vp],
            "mlora_base_gemm": [vp, vp, vp, i32, i32, i32, vp],
            "mlora_lora_shrink": [vp, vp, vp, vp],
            "mlora_lora_expand": [vp, vp, vp, vp],
            "mlora_trace_enable": [i32],
            "mlora_trace_disable": [],
            "mlora_trace_read": [i32, vp, vp],
            "mlora_lora_apply_noalloc": [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp],
            "mlora_set_gemm_tile_n": [i32],
            "mlora_set_skinny_form": [i32],
            "mlora_check_wait_timeout": [vp],
            "mlora_load_adapter_sliced": [vp, i32, i32, vp, vp, vp, i32, f32, i32],
            "mlora_slot_cache_create": [i32, vp],
            "mlora_slot_cache_destroy": [vp],
            "mlora_slot_cache_assign": [vp, vp, i32, vp, vp, vp, vp],
            "mlora_slot_cache_lookup": [vp, ctypes.c_int64, vp],
            "mlora_slot_cache_pin": [vp, ctypes.c_int64, i32],
            "mlora_slot_cache_evict": [vp, ctypes.c_int64],
            "mlora_adapter_cache_create": [vp, i32, vp],
            "mlora_adapter_cache_destroy": [vp],
            "mlora_adapter_cache_register": [vp, ctypes.c_int64, vp, vp, i32, f32, i32],
            "mlora_adapter_cache_unregister": [vp, ctypes.c_int64],
            "mlora_adapter_cache_pin": [vp, ctypes.c_int64, i32],
            "mlora_adapter_cache_map": [vp, vp, i32, vp, vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = i32
        lib.mlora_pool_bytes.argtypes = [i32, i32, i32, i32]
        lib.mlora_pool_bytes.restype = ctypes.c_size_t
        lib.mlora_status_string.argtypes = [i32]
        lib.mlora_status_string.restype = ctypes.c_char_p
        lib.mlora_last_error.argtypes = []
        lib.mlora_last_error.restype = ctypes.c_char_p
        lib.mlora_version.argtypes = []
        lib.mlora_version.restype = i32
        lib.mlora_launch_count.argtypes = []
        lib.mlora_launch_count.restype = u64
        lib.mlora_kernel_kind_name.argtypes = [i32]
        lib.mlora_kernel_kind_name.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _check(status: int, fn: str):
    if status != MLORA_OK:
        raise MloraError(status, fn, _lib.mlora_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------------- pool
def mlora_pool_create(n_slots: int, r_max: int, K: int, D: int, copy_stream=None) -> int:
    lib = load()
    out = ctypes.c_void_p()
    _check(lib.mlora_pool_create(n_slots, r_max, K, D, _stream(copy_stream), ctypes.byref(out)), "mlora_pool_create")
    return out.value


def mlora_pool_create_classes(class_slots, class_rank, K: int, D: int, copy_stream=None) -> int:
    """A pool whose slots come in rank classes: class c has class_slots[c] slots of rank <= class_rank[c]."""
    lib = load()
    n = len(class_slots)
    assert len(class_rank) == n
    cs = (ctypes.c_int * n)(*[int(v) for v in class_slots])
    cr = (ctypes.c_int * n)(*[int(v) for v in class_rank])
    out = ctypes.c_void_p()
    _check(lib.mlora_pool_create_classes(n, cs, cr, K, D, _stream(copy_stream), ctypes.byref(out)),
           "mlora_pool_create_classes")
    return out.value


def mlora_embedding_pool_create(class_slots, class_rank, vocab: int, dim: int, copy_stream=None) -> int:
    """The slot pool of an embedding table [vocab, dim]: class c has class_slots[c] slots of rank <= class_rank[c]."""
    lib = load()
    n = len(class_slots)
    assert len(class_rank) == n
    cs = (ctypes.c_int * n)(*[int(v) for v in class_slots])
    cr = (ctypes.c_int * n)(*[int(v) for v in class_rank])
    out = ctypes.c_void_p()
    _check(lib.mlora_embedding_pool_create(n, cs, cr, vocab, dim, _stream(copy_stream), ctypes.byref(out)),
           "mlora_embedding_pool_create")
    return out.value


def mlora_pool_layout(pool: int, n_slots: int) -> dict:
    """The pool's column space: C and each slot's first column and width."""
    c = ctypes.c_int()
    off = (ctypes.c_int32 * n_slots)()
    width = (ctypes.c_int32 * n_slots)()
    _check(load().mlora_pool_layout(pool, ctypes.byref(c), off, width), "mlora_pool_layout")
    return dict(C=c.value, slot_off=list(off), slot_width=list(width))


def mlora_pool_destroy(pool: int) -> None:
    _check(load().mlora_pool_destroy(pool), "mlora_pool_destroy")


def mlora_load_adapter(pool: int, slot: int, A_host, B_host, rank: int, alpha: float, rslora: bool) -> None:
    """A_host [rank, K] and B_host [D, rank]: host bf16 (uint16 numpy arrays or CPU torch tensors)."""
    a, b = _host_ptr(A_host), _host_ptr(B_host)
    _check(load().mlora_load_adapter(pool, slot, a, b, rank, float(alpha), int(bool(rslora))), "mlora_load_adapter")


def mlora_load_adapter_sliced(pool: int, slot: int, A_slices, B_slices, rank: int, alpha: float,
                              rslora: bool) -> None:
    """Per-slice adapter of a fused linear: A_slices[i] [rank, K], B_slices[i] [width_i, rank] host
    bf16 (uint16 numpy arrays or CPU torch tensors); the widths are the B slices' row counts."""
    n = len(A_slices)
    assert len(B_slices) == n
    widths = (ctypes.c_int * n)(*[int(b.shape[0]) for b in B_slices])
    a_ptrs = (ctypes.c_void_p * n)(*[_host_ptr(a) for a in A_slices])
    b_ptrs = (ctypes.c_void_p * n)(*[_host_ptr(b) for b in B_slices])
    _check(load().mlora_load_adapter_sliced(pool, slot, n, widths, a_ptrs, b_ptrs, rank, float(alpha),
                                            int(bool(rslora))), "mlora_load_adapter_sliced")


def mlora_clear_slot(pool: int, slot: int) -> None:
    _check(load().mlora_clear_slot(pool, slot), "mlora_clear_slot")


def mlora_pool_sync(pool: int) -> None:
    _check(load().mlora_pool_sync(pool), "mlora_pool_sync")


def mlora_pool_info(pool: int) -> dict:
    i = [ctypes.c_int() for _ in range(4)]
    p = [ctypes.c_void_p() for _ in range(4)]
    _check(load().mlora_pool_info(pool, *(ctypes.byref(v) for v in i), *(ctypes.byref(v) for v in p)),
           "mlora_pool_info")
    return dict(n_slots=i[0].value, r_pad=i[1].value, K=i[2].value, D=i[3].value, A_pool=p[0].value,
                B_pool=p[1].value, slot_scale=p[2].value, slot_rank=p[3].value)


def mlora_pool_bytes(n_slots: int, r_max: int, K: int, D: int) -> int:
    return int(load().mlora_pool_bytes(n_slots, r_max, K, D))


# ------------------------------------------------------------------------- meta
def mlora_meta_create(max_tokens: int, max_slots_per_token: int, r_max: int) -> int:
    out = ctypes.c_void_p()
    _check(load().mlora_meta_create(max_tokens, max_slots_per_token, r_max, ctypes.byref(out)), "mlora_meta_create")
    return out.value


def mlora_meta_destroy(meta: int) -> None:
    _check(load().mlora_meta_destroy(meta), "mlora_meta_destroy")


def mlora_build_meta(meta: int, token_slots, scales, T: int, J: int, pool: int, stream=None) -> None:
    _check(load().mlora_build_meta(meta, _ptr(token_slots), _ptr(scales), T, J, pool, _stream(stream)),
           "mlora_build_meta")


def mlora_meta_status(meta: int) -> None:
    _check(load().mlora_meta_status(meta), "mlora_meta_status")


def mlora_meta_status_code(meta: int) -> int:
    return int(load().mlora_meta_status(meta))


def mlora_meta_read(meta: int, n_pairs: int) -> dict:
    import numpy as np
    order = np.zeros(max(n_pairs, 1), dtype=np.int32)
    seg_slot = np.zeros(n_pairs + 2, dtype=np.int32)
    seg_off = np.zeros(n_pairs + 2, dtype=np.int32)
    n_seg, n_active = ctypes.c_int(), ctypes.c_int()
    _check(load().mlora_meta_read(meta, order.ctypes.data, seg_slot.ctypes.data, seg_off.ctypes.data,
                                  ctypes.byref(n_seg), ctypes.byref(n_active)), "mlora_meta_read")
    k = n_seg.value
    return dict(order=order[:n_pairs].tolist(), seg_slot=seg_slot[:k].tolist(), seg_off=seg_off[:k + 1].tolist(),
                n_active=n_active.value)


# ------------------------------------------------------------------------- layer
def mlora_linear(pool: int, meta: int, x, W, y, stream=None) -> None:
    _check(load().mlora_linear(pool, meta, _ptr(x), _ptr(W), _ptr(y), _stream(stream)), "mlora_linear")


def mlora_embedding(pool: int, meta: int, ids, E, y, stream=None) -> None:
    """y[t] = E[ids[t]] + the step's LoRA side path on the lookup (ids int32 [T], E bf16 [vocab, dim], y fp32 [T, dim])."""
    _check(load().mlora_embedding(pool, meta, _ptr(ids), _ptr(E), _ptr(y), _stream(stream)), "mlora_embedding")


def mlora_base_gemm(x, W, y, T: int, K: int, D: int, stream=None) -> None:
    _check(load().mlora_base_gemm(_ptr(x), _ptr(W), _ptr(y), T, K, D, _stream(stream)), "mlora_base_gemm")


def mlora_lora_shrink(pool: int, meta: int, x, stream=None) -> None:
    _check(load().mlora_lora_shrink(pool, meta, _ptr(x), _stream(stream)), "mlora_lora_shrink")


def mlora_lora_expand(pool: int, meta: int, y, stream=None) -> None:
    _check(load().mlora_lora_expand(pool, meta, _ptr(y), _stream(stream)), "mlora_lora_expand")


def mlora_lora_apply_noalloc(x, y, token_slots, scales, T: int, J: int, A_pool, B_pool, slot_scale, slot_rank,
                             n_slots: int, r_pad: int, K: int, D: int, stream=None) -> None:
    """y += the LoRA side path, using only the caller's buffers and the library's built-in workspace."""
    _check(load().mlora_lora_apply_noalloc(_ptr(x), _ptr(y), _ptr(token_slots), _ptr(scales), T, J, _ptr(A_pool),
                                           _ptr(B_pool), _ptr(slot_scale), _ptr(slot_rank), n_slots, r_pad, K, D,
                                           _stream(stream)), "mlora_lora_apply_noalloc")


def mlora_set_path(path: int) -> None:
    """0 automatic, 1 the small-batch path whenever allowed, 2 always the tensor-core side path."""
    _check(load().mlora_set_path(path), "mlora_set_path")


def mlora_set_gemm_tile_n(n: int) -> None:
    """0 automatic, -1 never the CTA-pair GEMM, 256/224/192/128 always it with that N tile."""
    _check(load().mlora_set_gemm_tile_n(n), "mlora_set_gemm_tile_n")


def mlora_set_skinny_form(form: int) -> None:
    """Small-batch GEMM form: 0 and 1 split-K (CTA pairs), 2 token-split whenever it fits one wave."""
    _check(load().mlora_set_skinny_form(form), "mlora_set_skinny_form")


# ------------------------------------------------------------------------- slot residency
def mlora_slot_cache_create(n_slots: int) -> int:
    out = ctypes.c_void_p()
    _check(load().mlora_slot_cache_create(n_slots, ctypes.byref(out)), "mlora_slot_cache_create")
    return out.value


def mlora_slot_cache_destroy(cache: int) -> None:
    _check(load().mlora_slot_cache_destroy(cache), "mlora_slot_cache_destroy")


def mlora_slot_cache_assign(cache: int, ids) -> tuple:
    """(slots [n] int32, loads [(id, slot), ...]) for one step's adapter ids (-1 = none)."""
    import numpy as np
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int64).ravel())
    n = len(ids)
    slots = np.zeros(max(n, 1), np.int32)
    load_ids = np.zeros(max(n, 1), np.int64)
    load_slots = np.zeros(max(n, 1), np.int32)
    n_loads = ctypes.c_int()
    _check(load().mlora_slot_cache_assign(cache, ids.ctypes.data, n, slots.ctypes.data, load_ids.ctypes.data,
                                          load_slots.ctypes.data, ctypes.byref(n_loads)), "mlora_slot_cache_assign")
    k = n_loads.value
    return slots[:n], list(zip(load_ids[:k].tolist(), load_slots[:k].tolist()))


def mlora_slot_cache_lookup(cache: int, adapter_id: int) -> int:
    out = ctypes.c_int32()
    _check(load().mlora_slot_cache_lookup(cache, adapter_id, ctypes.byref(out)), "mlora_slot_cache_lookup")
    return out.value


def mlora_slot_cache_pin(cache: int, adapter_id: int, pinned: bool = True) -> None:
    _check(load().mlora_slot_cache_pin(cache, adapter_id, int(bool(pinned))), "mlora_slot_cache_pin")


def mlora_slot_cache_evict(cache: int, adapter_id: int) -> None:
    _check(load().mlora_slot_cache_evict(cache, adapter_id), "mlora_slot_cache_evict")


def mlora_adapter_cache_create(pools) -> int:
    arr = (ctypes.c_void_p * len(pools))(*pools)
    out = ctypes.c_void_p()
    _check(load().mlora_adapter_cache_create(arr, len(pools), ctypes.byref(out)), "mlora_adapter_cache_create")
    return out.value


def mlora_adapter_cache_destroy(cache: int) -> None:
    _check(load().mlora_adapter_cache_destroy(cache), "mlora_adapter_cache_destroy")


def mlora_adapter_cache_register(cache: int, adapter_id: int, A_host, B_host, rank: int, alpha: float,
                                 rslora: bool) -> None:
    """A_host / B_host: one host bf16 buffer per pool (kept alive by the caller while registered)."""
    a = (ctypes.c_void_p * len(A_host))(*[_host_ptr(x) for x in A_host])
    b = (ctypes.c_void_p * len(B_host))(*[_host_ptr(x) for x in B_host])
    _check(load().mlora_adapter_cache_register(cache, adapter_id, a, b, rank, float(alpha), int(bool(rslora))),
           "mlora_adapter_cache_register")


def mlora_adapter_cache_unregister(cache: int, adapter_id: int) -> None:
    _check(load().mlora_adapter_cache_unregister(cache, adapter_id), "mlora_adapter_cache_unregister")


def mlora_adapter_cache_pin(cache: int, adapter_id: int, pinned: bool = True) -> None:
    _check(load().mlora_adapter_cache_pin(cache, adapter_id, int(bool(pinned))), "mlora_adapter_cache_pin")


def mlora_adapter_cache_map(cache: int, ids) -> tuple:
    """(token_slots [n] int32 host array, number of adapters loaded) for one step's adapter ids."""
    import numpy as np
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int64).ravel())
    slots = np.zeros(max(len(ids), 1), np.int32)
    n_loaded = ctypes.c_int()
    _check(load().mlora_adapter_cache_map(cache, ids.ctypes.data, len(ids), slots.ctypes.data,
                                          ctypes.byref(n_loaded)), "mlora_adapter_cache_map")
    return slots[:len(ids)], n_loaded.value


# ------------------------------------------------------------------------- diagnostics
def mlora_check_wait_timeout(stream=None) -> int:
    """Status of the bounded-wait check (MLORA_ERR_DEVICE_TIMEOUT is the expected result)."""
    return int(load().mlora_check_wait_timeout(_stream(stream)))


def mlora_status_string(status: int) -> str:
    return load().mlora_status_string(status).decode()


def mlora_last_error() -> str:
    return load().mlora_last_error().decode(errors="replace")


def mlora_version() -> int:
    return int(load().mlora_version())


def mlora_launch_count() -> int:
    return int(load().mlora_launch_count())


def mlora_trace_enable(capacity: int = 4096) -> None:
    _check(load().mlora_trace_enable(capacity), "mlora_trace_enable")


def mlora_trace_disable() -> None:
    _check(load().mlora_trace_disable(), "mlora_trace_disable")


def mlora_trace_read() -> dict:
    n = len(KERNEL_KINDS)
    launches = (ctypes.c_int * n)()
    ms = (ctypes.c_double * n)()
    _check(load().mlora_trace_read(n, launches, ms), "mlora_trace_read")
    return {KERNEL_KINDS[k]: (launches[k], ms[k]) for k in range(n)}


def mlora_kernel_kind_name(kind: int) -> str:
    return load().mlora_kernel_kind_name(kind).decode()


def _host_ptr(a) -> int:
    import numpy as np
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16 and a.flags.c_contiguous
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        assert not a.is_cuda and a.is_contiguous()
        return a.data_ptr()
    if isinstance(a, int):
        return a
    raise TypeError(type(a))
