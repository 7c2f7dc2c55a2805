"""Seeded synthetic inputs for the multi-LoRA linear layer (shared by the oracle and the CUDA path).

This module draws random numbers and lays out the workloads; it contains none of
the layer's arithmetic (no scaling factor, no product, no sort). Everything is
keyed by (seed, tensor id, element index) through the counter-based generator in
``philox_normal.c``, so any slice of any tensor can be regenerated alone.

The workload recipes follow the shapes and distributions that the pages give:
- "Multi-LoRA Serving Explained" (sevydevy.com), sections on the weight-matrix
  maths and the stacked slot pool: hidden 4096, MLP 14336, ranks 8/16/64.
- "[RFC] Per-request activation of multiple LoRA adapters" (vLLM issue 51940),
  "Proposed Change": k adapters per request, per-adapter scales, sentinel fill.
- "[vLLM] LoRA" (secrett2633 blog), PEFTHelper: rsLoRA flag per adapter.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox_normal.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_lock = threading.Lock()

SEED_BASE = 0x6D4C6F52


def build(force: bool = False) -> str:
    """Compile the generator with gcc (host code only, no -march, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.synth_philox4x64_10.argtypes = [vp, vp, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
            lib.synth_normal_f64.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
            lib.synth_u64.argtypes = [u64, u64, u64, u64, vp, i32]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def philox4x64_10(counter, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.zeros(4, dtype=np.uint64)
    _load().synth_philox4x64_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def tensor_key(*parts: int) -> int:
    """Pack small non-negative ints (each < 2^12, at most 5) into one 64-bit tensor id."""
    key = 0
    assert len(parts) <= 5
    for p in parts:
        assert 0 <= p < (1 << 12), p
        key = (key << 12) | int(p)
    return key | (len(parts) << 60)


def normal_bf16(seed: int, tid: int, shape, std: float = 1.0, first: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of std * N(0,1), elements [first, first + prod(shape))."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, tid, first, n, float(std), out.ctypes.data, _threads())
    return out.reshape(shape)


def normal_f64(seed: int, tid: int, shape, std: float = 1.0, first: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    if n:
        _load().synth_normal_f64(seed, tid, first, n, float(std), out.ctypes.data, _threads())
    return out.reshape(shape)


def raw_u64(seed: int, tid: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.uint64)
    if n:
        _load().synth_u64(seed, tid, first, int(n), out.ctypes.data, _threads())
    return out


def uniform01(seed: int, tid: int, n: int) -> np.ndarray:
    """Uniform [0, 1) doubles from the top 53 bits of each word."""
    return (raw_u64(seed, tid, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------
# Workload recipes
# --------------------------------------------------------------------------------------

# tensor-id namespaces (first packed field)
_NS_W, _NS_X, _NS_A, _NS_B, _NS_SLOTS, _NS_SCALES, _NS_MISC = 1, 2, 3, 4, 5, 6, 7


@dataclass
class Adapter:
    """One LoRA adapter for one linear: A [rank, K], B [D, rank] as bf16 bits."""
    A: np.ndarray
    B: np.ndarray
    rank: int
    alpha: float
    rslora: bool = False


@dataclass
class Linear:
    name: str
    K: int
    D: int
    W: np.ndarray | None            # [D, K] bf16 bits (None when generated lazily by rows)
    x_id: int                       # which activation matrix feeds it
    adapters: dict = field(default_factory=dict)   # slot -> Adapter


@dataclass
class Workload:
    name: str
    seed: int
    T: int
    J: int
    n_slots: int
    r_max: int
    token_slots: np.ndarray         # [T, J] int32, -1 = no adapter
    scales: np.ndarray | None       # [T, J] float32 or None (= 1)
    xs: dict                        # x_id -> [T, K] bf16 bits
    linears: list
    notes: str = ""
    phases: list = field(default_factory=list)   # (name, first token, end token) sub-batches
    classes: list | None = None     # [(slots, rank), ...] rank classes of the pools (None: one class)


def _adapter(seed, layer, module, adapter_id, K, D, rank, alpha, rslora, std=0.02):
    A = normal_bf16(seed, tensor_key(_NS_A, layer, module, adapter_id), (rank, K), std)
    B = normal_bf16(seed, tensor_key(_NS_B, layer, module, adapter_id), (D, rank), std)
    return Adapter(A=A, B=B, rank=rank, alpha=float(alpha), rslora=bool(rslora))


def tiny(T: int = 16, K: int = 256, D: int = 256, n_adapters: int = 4, rank: int = 8,
         alpha: float = 16.0, seed_offset: int = 1) -> Workload:
    """One linear d=k=256, bf16 W ~ N(0, 0.02); 4 adapters of rank 8 (A, B ~ N(0, 0.02), alpha 16);
    16 tokens of x ~ N(0, 1); per-token slot uniform over {-1, 0, 1, 2, 3}; k = 1, s = 1."""
    seed = SEED_BASE + seed_offset
    slots = (raw_u64(seed, tensor_key(_NS_SLOTS), T) % np.uint64(n_adapters + 1)).astype(np.int64) - 1
    lin = Linear("linear", K, D, normal_bf16(seed, tensor_key(_NS_W, 0, 0), (D, K), 0.02), 0)
    for s in range(n_adapters):
        lin.adapters[s] = _adapter(seed, 0, 0, s, K, D, rank, alpha, False)
    return Workload("tiny", seed, T, 1, n_adapters, rank,
                    slots.astype(np.int32).reshape(T, 1), None,
                    {0: normal_bf16(seed, tensor_key(_NS_X, 0), (T, K), 1.0)}, [lin])


def decode(T: int = 256, hidden: int = 4096, n_adapters: int = 100, rank: int = 16,
           alpha: float = 32.0, p_sentinel: float = 0.1, modules=("q", "k", "v", "o"),
           seed_offset: int = 2) -> Workload:
    """Decode batch: T tokens at hidden 4096 through q/k/v/o-shaped 4096->4096 linears; 100 resident
    adapters of rank 16 (alpha 32) per linear; per-token slot uniform over the 100, with a 10 %
    chance of the sentinel -1. q, k and v read the same x, o reads a second one."""
    seed = SEED_BASE + seed_offset
    u = uniform01(seed, tensor_key(_NS_SLOTS, 0), T)
    pick = (raw_u64(seed, tensor_key(_NS_SLOTS, 1), T) % np.uint64(n_adapters)).astype(np.int64)
    slots = np.where(u < p_sentinel, -1, pick).astype(np.int32).reshape(T, 1)
    linears = []
    for m, name in enumerate(modules):
        lin = Linear(name, hidden, hidden,
                     normal_bf16(seed, tensor_key(_NS_W, 0, m), (hidden, hidden), 0.02),
                     1 if name == "o" else 0)
        for s in range(n_adapters):
            lin.adapters[s] = _adapter(seed, 0, m, s, hidden, hidden, rank, alpha, False)
        linears.append(lin)
    xs = {0: normal_bf16(seed, tensor_key(_NS_X, 0), (T, hidden), 1.0)}
    if any(l.x_id == 1 for l in linears):
        xs[1] = normal_bf16(seed, tensor_key(_NS_X, 1), (T, hidden), 1.0)
    return Workload("decode", seed, T, 1, n_adapters, rank, slots, None, xs, linears)


def prefill(n_requests: int = 8, seg_len: int = 512, hidden: int = 4096, mlp: int = 14336,
            ranks=(8, 16, 64), r_max: int = 64, seed_offset: int = 3, lazy_w: bool = False) -> Workload:
    """Prefill batch: 8 requests of 512 contiguous tokens, request i on slot i; fused gate_up
    4096 -> 2*14336 and down 14336 -> 4096; ranks cycle 8/16/64 padded to r_max 64; alpha = 2r."""
    seed = SEED_BASE + seed_offset
    T = n_requests * seg_len
    slots = np.repeat(np.arange(n_requests, dtype=np.int32), seg_len).reshape(T, 1)
    shapes = [("gate_up", hidden, 2 * mlp, 0), ("down", mlp, hidden, 1)]
    linears = []
    for m, (name, K, D, xid) in enumerate(shapes):
        W = None if lazy_w else normal_bf16(seed, tensor_key(_NS_W, 0, m), (D, K), 0.02)
        lin = Linear(name, K, D, W, xid)
        for s in range(n_requests):
            r = ranks[s % len(ranks)]
            lin.adapters[s] = _adapter(seed, 0, m, s, K, D, r, 2.0 * r, False)
        linears.append(lin)
    xs = {0: normal_bf16(seed, tensor_key(_NS_X, 0), (T, hidden), 1.0),
          1: normal_bf16(seed, tensor_key(_NS_X, 1), (T, mlp), 1.0)}
    return Workload("prefill", seed, T, 1, n_requests, r_max, slots, None, xs, linears)


def compose(T: int = 128, hidden: int = 4096, qkv_out: int = 6144, n_adapters: int = 32,
            rank: int = 16, alpha: float = 32.0, J: int = 3, seed_offset: int = 4) -> Workload:
    """Multi-adapter decode: T tokens, qkv 4096 -> 6144; each token draws n ~ U{1..J} adapters
    without replacement from 32 rank-16 adapters, trailing slots -1; per-request scales
    U[0.2, 1.0] (fp32); adapters with an even slot id use rsLoRA."""
    seed = SEED_BASE + seed_offset
    n_act = (raw_u64(seed, tensor_key(_NS_SLOTS, 0), T) % np.uint64(J)).astype(np.int64) + 1
    words = raw_u64(seed, tensor_key(_NS_SLOTS, 1), T * J).reshape(T, J)
    slots = np.full((T, J), -1, dtype=np.int32)
    for t in range(T):
        pool = list(range(n_adapters))
        for j in range(int(n_act[t])):          # partial Fisher-Yates, without replacement
            i = j + int(words[t, j] % np.uint64(n_adapters - j))
            pool[j], pool[i] = pool[i], pool[j]
            slots[t, j] = pool[j]
    u = uniform01(seed, tensor_key(_NS_SCALES, 0), T * J).reshape(T, J)
    scales = (0.2 + 0.8 * u).astype(np.float32)
    scales[slots < 0] = 0.0
    lin = Linear("qkv", hidden, qkv_out,
                 normal_bf16(seed, tensor_key(_NS_W, 0, 0), (qkv_out, hidden), 0.02), 0)
    for s in range(n_adapters):
        lin.adapters[s] = _adapter(seed, 0, 0, s, hidden, qkv_out, rank, alpha, s % 2 == 0)
    xs = {0: normal_bf16(seed, tensor_key(_NS_X, 0), (T, hidden), 1.0)}
    return Workload("compose", seed, T, J, n_adapters, rank, slots, scales, xs, [lin])


def logits(T: int = 256, hidden: int = 4096, vocab: int = 128256, n_adapters: int = 16,
           ranks: tuple = (8, 16, 32), J: int = 2, sentinel_frac: float = 0.1,
           seed_offset: int = 6) -> Workload:
    """The side path on the LM head with router-weighted mixtures: T decode tokens through the
    hidden -> vocab linear (Llama-3-sized vocabulary by default); every token mixes J distinct
    adapters drawn without replacement from n_adapters, weighted by per-token gate values (a
    softmax over J router logits drawn N(0, 1), as a learned per-token router would emit);
    sentinel_frac of the tokens use no adapter. Adapter i has rank ranks[i % len(ranks)] and
    alpha = 2r; the pool's rank width is max(ranks)."""
    seed = SEED_BASE + seed_offset
    words = raw_u64(seed, tensor_key(_NS_SLOTS, 0), T * J).reshape(T, J)
    none = uniform01(seed, tensor_key(_NS_SLOTS, 1), T) < sentinel_frac
    slots = np.full((T, J), -1, dtype=np.int32)
    for t in range(T):
        if none[t]:
            continue
        pool = list(range(n_adapters))
        for j in range(J):                      # partial Fisher-Yates, without replacement
            i = j + int(words[t, j] % np.uint64(n_adapters - j))
            pool[j], pool[i] = pool[i], pool[j]
            slots[t, j] = pool[j]
    z = normal_f64(seed, tensor_key(_NS_SCALES, 0), (T, J))
    g = np.exp(z - z.max(axis=1, keepdims=True))
    scales = (g / g.sum(axis=1, keepdims=True)).astype(np.float32)
    scales[slots < 0] = 0.0
    r_max = max(ranks)
    lin = Linear("lm_head", hidden, vocab, normal_bf16(seed, tensor_key(_NS_W, 0, 0), (vocab, hidden), 0.02), 0)
    for s in range(n_adapters):
        r = ranks[s % len(ranks)]
        lin.adapters[s] = _adapter(seed, 0, 0, s, hidden, vocab, r, 2.0 * r, False)
    xs = {0: normal_bf16(seed, tensor_key(_NS_X, 0), (T, hidden), 1.0)}
    return Workload("logits", seed, T, J, n_adapters, r_max, slots, scales, xs, [lin])


def zipf_admission(n_requests: int, n_ids: int, exponent: float, max_distinct: int,
                   seed: int, tid: int, class_of=None, class_cap=None) -> list:
    """Draw request tenants from Zipf(exponent) over ids 1..n_ids and admit them in order: a
    request whose adapter is new is deferred when the batch already holds max_distinct adapters
    (the max-loras admission rule) or, with class_of / class_cap, when the adapter's rank class
    already holds class_cap[class_of(id)] adapters. Returns the admitted ids in admission order."""
    w = 1.0 / np.arange(1, n_ids + 1, dtype=np.float64) ** exponent
    cdf = np.cumsum(w) / w.sum()
    admitted, distinct, i = [], [], 0
    per_class = {}
    u = uniform01(seed, tid, 64 * n_requests + 64)
    while len(admitted) < n_requests and i < len(u):
        a = int(np.searchsorted(cdf, u[i], side="right")) + 1
        i += 1
        if a not in distinct:
            if len(distinct) >= max_distinct:
                continue
            if class_cap is not None:
                c = class_of(a)
                if per_class.get(c, 0) >= class_cap[c]:
                    continue
                per_class[c] = per_class.get(c, 0) + 1
            distinct.append(a)
        admitted.append(a)
    return admitted


MIXED_RANKS = (8, 16, 64)


def mixed_class_slots(n_slots: int = 128, n_registered: int = 1000) -> list:
    """Slots per rank class of the mixed step's pools: n_slots split in proportion to the
    registered adapters of each rank (rank of id a = MIXED_RANKS[a mod 3]), largest remainder."""
    counts = [sum(1 for a in range(1, n_registered + 1) if a % 3 == c) for c in range(3)]
    quota = [n_slots * c / n_registered for c in counts]
    out = [int(q) for q in quota]
    for c in sorted(range(3), key=lambda c: (-(quota[c] - out[c]), c))[:n_slots - sum(out)]:
        out[c] += 1
    return out


def mixed_step_plan(n_prefill: int = 4, prefill_len: int = 192, n_decode: int = 256,
                    n_registered: int = 1000, n_slots: int = 128, zipf: float = 1.1,
                    seed_offset: int = 5, classes: bool = True):
    """Mixed serving step: 4 prefill segments of 192 tokens (one request each) then 256 decode
    tokens (one request each); tenants Zipf(1.1) over 1000 registered ids; rank by id is
    [8, 16, 64][id mod 3], alpha = 2r. With classes (default) the 128 slots form three rank
    classes (8, 16, 64) sized by mixed_class_slots, a new adapter is admitted only while its
    class has a free slot, and class c's adapters take its slots in first-seen order (slots are
    numbered class by class); without, any adapter takes the next of 128 slots of rank 64."""
    seed = SEED_BASE + seed_offset
    class_of = lambda a: a % 3  # noqa: E731
    sizes = mixed_class_slots(n_slots, n_registered) if classes else None
    tenants = zipf_admission(n_prefill + n_decode, n_registered, zipf, n_slots, seed,
                             tensor_key(_NS_MISC, 0), class_of=class_of if classes else None, class_cap=sizes)
    slot_of = {}
    if classes:
        base = [0, sizes[0], sizes[0] + sizes[1]]
        used = [0, 0, 0]
        for a in tenants:
            if a not in slot_of:
                c = class_of(a)
                slot_of[a] = base[c] + used[c]
                used[c] += 1
    else:
        for a in tenants:
            slot_of.setdefault(a, len(slot_of))
    per_token = []
    for i, a in enumerate(tenants):
        per_token += [slot_of[a]] * (prefill_len if i < n_prefill else 1)
    T = len(per_token)
    ranks = {a: MIXED_RANKS[a % 3] for a in slot_of}
    return dict(seed=seed, T=T, token_slots=np.array(per_token, dtype=np.int32).reshape(T, 1),
                slot_of=slot_of, rank_of=ranks, tenants=tenants,
                classes=[(sizes[c], MIXED_RANKS[c]) for c in range(3)] if classes else None,
                n_prefill_tokens=n_prefill * prefill_len)


MIXED_MODULES = (("qkv", 4096, 6144, 0), ("o", 4096, 4096, 1),
                 ("gate_up", 4096, 28672, 2), ("down", 14336, 4096, 3))


def mixed_adapter(seed: int, layer: int, module: int, adapter_id: int, K: int, D: int) -> Adapter:
    r = MIXED_RANKS[adapter_id % 3]
    return _adapter(seed, layer, module, adapter_id, K, D, r, 2.0 * r, False)


def mixed_weight_rows(seed: int, layer: int, module: int, K: int, row0: int, n_rows: int) -> np.ndarray:
    return normal_bf16(seed, tensor_key(_NS_W, layer, module), (n_rows, K), 0.02, first=row0 * K)


def mixed_x(seed: int, layer: int, module: int, T: int, K: int) -> np.ndarray:
    return normal_bf16(seed, tensor_key(_NS_X, layer, module), (T, K), 1.0)


@dataclass
class LazyAdapter:
    """An adapter of the mixed step known by its id; A and B are generated on demand."""
    seed: int
    layer: int
    module: int
    adapter_id: int
    rank: int
    alpha: float
    rslora: bool = False

    def materialize(self, K: int, D: int) -> Adapter:
        return mixed_adapter(self.seed, self.layer, self.module, self.adapter_id, K, D)


def mixed(n_layers: int = 32, classes: bool = True) -> Workload:
    """The mixed serving step as a workload whose tensors are generated on demand: linears
    layer-major over MIXED_MODULES (x_id = linear index), adapters as LazyAdapter, W = None and
    no xs entries (see materialize_linear / materialize_x). With classes (default) the pools'
    128 slots come in rank classes 8 / 16 / 64 (mixed_step_plan)."""
    plan = mixed_step_plan(classes=classes)
    seed = plan["seed"]
    linears = []
    for l in range(n_layers):
        for m, (name, K, D, _) in enumerate(MIXED_MODULES):
            lin = Linear(f"L{l}.{name}", K, D, None, len(linears))
            for a, s in plan["slot_of"].items():
                r = plan["rank_of"][a]
                lin.adapters[s] = LazyAdapter(seed, l, m, a, r, 2.0 * r, False)
            linears.append(lin)
    n_pre = plan["n_prefill_tokens"]
    return Workload("mixed", seed, plan["T"], 1, 128, 64, plan["token_slots"], None, {}, linears,
                    notes="tensors generated on demand by layer and module",
                    phases=[("prefill", 0, n_pre), ("decode", n_pre, plan["T"])], classes=plan["classes"])


def _layer_module(wl: Workload, lin: Linear) -> tuple:
    return lin.x_id // len(MIXED_MODULES), lin.x_id % len(MIXED_MODULES)


def materialize_linear(wl: Workload, lin: Linear) -> Linear:
    """lin with W and its adapters generated (a no-op for an eager linear)."""
    if lin.W is not None:
        return lin
    l, m = _layer_module(wl, lin)
    out = Linear(lin.name, lin.K, lin.D, mixed_weight_rows(wl.seed, l, m, lin.K, 0, lin.D), lin.x_id)
    out.adapters = {s: a.materialize(lin.K, lin.D) for s, a in lin.adapters.items()}
    return out


def materialize_x(wl: Workload, lin: Linear) -> np.ndarray:
    if lin.x_id in wl.xs:
        return wl.xs[lin.x_id]
    l, m = _layer_module(wl, lin)
    return mixed_x(wl.seed, l, m, wl.T, lin.K)


def linear_weight(wl: Workload, lin: Linear) -> np.ndarray:
    """W of a linear, generated on demand for the mixed step."""
    if lin.W is not None:
        return lin.W
    l, m = _layer_module(wl, lin)
    return mixed_weight_rows(wl.seed, l, m, lin.K, 0, lin.D)


# --------------------------------------------------------------------------------------
# Embedding lookup with LoRA
# --------------------------------------------------------------------------------------

_NS_EMB = 8


@dataclass
class EmbeddingWorkload:
    """Token ids through an embedding table with LoRA adapters in rank-class slots."""
    name: str
    seed: int
    T: int
    J: int
    vocab: int
    dim: int
    ids: np.ndarray                 # [T] int32 in [0, vocab)
    token_slots: np.ndarray         # [T, J] int32, -1 = no adapter
    scales: np.ndarray | None       # [T, J] float32 or None (= 1)
    E: np.ndarray                   # [vocab, dim] bf16 bits
    adapters: dict                  # slot -> Adapter with A [rank, vocab], B [dim, rank]
    classes: list                   # [(slots, rank), ...]

    @property
    def n_slots(self) -> int:
        return sum(n for n, _ in self.classes)

    @property
    def r_max(self) -> int:
        return max(r for _, r in self.classes)


def _embedding_tensors(seed, vocab, dim, T):
    ids = (raw_u64(seed, tensor_key(_NS_EMB, 0), T) % np.uint64(vocab)).astype(np.int32)
    E = normal_bf16(seed, tensor_key(_NS_EMB, 1), (vocab, dim), 0.02)
    return ids, E


def _embedding_adapter(seed, adapter_id, vocab, dim, rank, alpha, rslora):
    A = normal_bf16(seed, tensor_key(_NS_EMB, 2, adapter_id), (rank, vocab), 0.02)
    B = normal_bf16(seed, tensor_key(_NS_EMB, 3, adapter_id), (dim, rank), 0.02)
    return Adapter(A=A, B=B, rank=rank, alpha=float(alpha), rslora=bool(rslora))


def embedding_step(vocab: int = 100000, dim: int = 4096) -> EmbeddingWorkload:
    """The mixed serving step's batch through the token embedding: the same 1024 tokens and token
    -> slot map (mixed_step_plan: 4 x 192 prefill + 256 decode tokens, 112 adapters admitted into
    128 slots in rank classes 8 / 16 / 64, alpha = 2r), token ids uniform over the vocabulary
    (100000 x 4096, the memory example's table), E ~ N(0, 0.02), A [r, vocab] and B [dim, r]
    ~ N(0, 0.02) per adapter id."""
    plan = mixed_step_plan()
    seed = plan["seed"]
    ids, E = _embedding_tensors(seed, vocab, dim, plan["T"])
    adapters = {s: _embedding_adapter(seed, a, vocab, dim, plan["rank_of"][a], 2.0 * plan["rank_of"][a], False)
                for a, s in plan["slot_of"].items()}
    return EmbeddingWorkload("embedding", seed, plan["T"], 1, vocab, dim, ids, plan["token_slots"], None, E,
                             adapters, plan["classes"])


def embedding_case(T: int, vocab: int, dim: int, J: int, classes, sentinel_frac: float = 0.15,
                   with_scales: bool = True, seed_offset: int = 20) -> EmbeddingWorkload:
    """A small embedding workload for parity tests: every slot of the classes holds an adapter
    (rank = its class's rank for the first slot of a class, else uniform in [1, class rank];
    alpha = 2r; odd slots rsLoRA); each token draws n ~ U{1..J} distinct slots (trailing -1),
    sentinel_frac of the tokens none; scales U[0.2, 1.0] or None."""
    seed = SEED_BASE + seed_offset
    n_slots = sum(n for n, _ in classes)
    ids, E = _embedding_tensors(seed, vocab, dim, T)
    rw = raw_u64(seed, tensor_key(_NS_EMB, 4), n_slots)
    adapters, s = {}, 0
    for n, r_cls in classes:
        for i in range(n):
            r = r_cls if i == 0 else 1 + int(rw[s] % np.uint64(r_cls))
            adapters[s] = _embedding_adapter(seed, s, vocab, dim, r, 2.0 * r, s % 2 == 1)
            s += 1
    n_act = (raw_u64(seed, tensor_key(_NS_SLOTS, 0), T) % np.uint64(J)).astype(np.int64) + 1
    none = uniform01(seed, tensor_key(_NS_SLOTS, 2), T) < sentinel_frac
    words = raw_u64(seed, tensor_key(_NS_SLOTS, 1), T * J).reshape(T, J)
    slots = np.full((T, J), -1, dtype=np.int32)
    for t in range(T):
        if none[t]:
            continue
        pool = list(range(n_slots))
        for j in range(min(int(n_act[t]), n_slots)):     # partial Fisher-Yates, without replacement
            k = j + int(words[t, j] % np.uint64(n_slots - j))
            pool[j], pool[k] = pool[k], pool[j]
            slots[t, j] = pool[j]
    scales = None
    if with_scales:
        u = uniform01(seed, tensor_key(_NS_SCALES, 0), T * J).reshape(T, J)
        scales = (0.2 + 0.8 * u).astype(np.float32)
        scales[slots < 0] = 0.0
    return EmbeddingWorkload("embedding_case", seed, T, J, vocab, dim, ids, slots, scales, E, adapters,
                             [(int(n), int(r)) for n, r in classes])
