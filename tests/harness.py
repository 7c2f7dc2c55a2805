"""Glue for GPU tests and the benchmark: puts a synthetic workload on the device through the
library's API, and compares device outputs with the fp64 oracle."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synth

# Tolerances for bf16 inputs with fp32 accumulation (per linear output tensor).
REL_FROB_TOL = 5e-3
MAX_ABS_TOL = 3e-2


def errors(y_dev: np.ndarray, y_ref: np.ndarray) -> tuple:
    diff = y_dev.astype(np.float64) - y_ref
    den = np.linalg.norm(y_ref)
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return rel, float(np.max(np.abs(diff))) if diff.size else 0.0


def assert_close(y_dev, y_ref, what: str, rel_tol: float = REL_FROB_TOL, abs_tol: float = MAX_ABS_TOL):
    rel, mx = errors(np.asarray(y_dev), np.asarray(y_ref))
    assert rel <= rel_tol and mx <= abs_tol, f"{what}: rel Frobenius {rel:.3e} (tol {rel_tol}), max abs {mx:.3e} (tol {abs_tol})"
    return rel, mx


@dataclass
class DeviceLinear:
    lin: synth.Linear
    pool: object
    W: object
    y: object


class DeviceWorkload:
    """A synth.Workload resident on the GPU: one pool per linear, W, x, token slots, scales."""

    def __init__(self, wl: synth.Workload, device="cuda:0", linears=None):
        import torch
        from rank_adapter_gemm_token_gb300 import layer

        self.torch = torch
        self.layer = layer
        self.wl = wl
        self.device = torch.device(device)
        self.meta = layer.StepMeta(max(wl.T, 1), wl.J, wl.r_max)
        self.token_slots = torch.from_numpy(np.ascontiguousarray(wl.token_slots.astype(np.int32))).to(self.device)
        self.scales = None if wl.scales is None else torch.from_numpy(
            np.ascontiguousarray(wl.scales.astype(np.float32))).to(self.device)
        self.x = {k: layer.bf16_from_bits(v, self.device) for k, v in wl.xs.items()}
        self.linears = []
        for lin in (wl.linears if linears is None else linears):
            lazy = lin.W is None                  # the mixed step: tensors generated here, per linear
            pool = layer.AdapterPool(wl.n_slots, wl.r_max, lin.K, lin.D, classes=getattr(wl, "classes", None))
            for s, ad in lin.adapters.items():
                if isinstance(ad, synth.LazyAdapter):
                    ad = ad.materialize(lin.K, lin.D)
                pool.load(s, ad.A, ad.B, ad.rank, ad.alpha, ad.rslora)
            if lazy:
                pool.sync()                       # release the pinned staging copies now
            W = layer.bf16_from_bits(synth.linear_weight(wl, lin), self.device)
            if lin.x_id not in self.x:
                self.x[lin.x_id] = layer.bf16_from_bits(synth.materialize_x(wl, lin), self.device)
            y = torch.empty((wl.T, lin.D), dtype=torch.float32, device=self.device)
            self.linears.append(DeviceLinear(lin, pool, W, y))
        for dl in self.linears:
            dl.pool.sync()

    def build_meta(self, stream=None):
        self.meta.build(self.token_slots, self.scales, self.linears[0].pool, stream)

    def run(self, stream=None):
        """One step: build the metadata once, then every linear of the workload."""
        self.build_meta(stream)
        for dl in self.linears:
            self.layer.linear(dl.pool, self.meta, self.x[dl.lin.x_id], dl.W, dl.y, stream)

    def sub_rows(self, r0: int, r1: int) -> "RowRange":
        """The same linears (pools, W) over token rows [r0, r1): a phase of the step."""
        return RowRange(self, r0, r1)

    def close(self):
        for dl in self.linears:
            dl.pool.close()
        self.meta.close()


class RowRange:
    """Token rows [r0, r1) of a DeviceWorkload through all of its linears, with metadata of their
    own (x and y are row slices of the workload's tensors)."""

    def __init__(self, dw: DeviceWorkload, r0: int, r1: int):
        self.dw, self.r0, self.r1 = dw, r0, r1
        self.meta = dw.layer.StepMeta(r1 - r0, dw.wl.J, dw.wl.r_max)
        self.token_slots = dw.token_slots[r0:r1].contiguous()
        self.scales = None if dw.scales is None else dw.scales[r0:r1].contiguous()

    def run(self, stream=None):
        dw = self.dw
        self.meta.build(self.token_slots, self.scales, dw.linears[0].pool, stream)
        for dl in dw.linears:
            dw.layer.linear(dl.pool, self.meta, dw.x[dl.lin.x_id][self.r0:self.r1], dl.W, dl.y[self.r0:self.r1],
                            stream)

    def close(self):
        self.meta.close()


def oracle_rows(wl: synth.Workload, lin: synth.Linear, rows=None, cols=None, threads=None) -> np.ndarray:
    return oracle.linear(wl.xs[lin.x_id], lin.W, wl.token_slots, lin.adapters, wl.n_slots, scales=wl.scales,
                         rows=rows, cols=cols, threads=threads)


def tile_rows(wl: synth.Workload, per_tile: int = 1, seed: int = 0) -> np.ndarray:
    """Token rows covering every 128-token tile (per_tile random rows each, plus the tile's
    first and last row) and the first token of every slot in use (sorted)."""
    rng = np.random.default_rng(seed)
    picks = set()
    for t0 in range(0, wl.T, 128):
        t1 = min(wl.T, t0 + 128)
        picks.update((t0, t1 - 1))
        picks.update(int(t) for t in rng.integers(t0, t1, size=per_tile))
    first = {}
    for t in range(wl.T):
        for s in wl.token_slots[t]:
            if s >= 0:
                first.setdefault(int(s), t)
    picks.update(first.values())
    return np.array(sorted(picks), dtype=np.int64)


def sample_rows(wl: synth.Workload, n: int, seed: int = 0) -> np.ndarray:
    """n token rows covering sentinel rows, both ends and a spread of slots (sorted)."""
    T = wl.T
    rng = np.random.default_rng(seed)
    picks = {0, T - 1}
    flat = wl.token_slots
    sent = np.where(np.all(flat < 0, axis=1))[0]
    if len(sent):
        picks.add(int(sent[0]))
    seen = set()
    for t in range(T):                       # first token of each distinct first slot
        s = int(flat[t, 0])
        if s not in seen and len(picks) < n // 2:
            seen.add(s)
            picks.add(t)
    while len(picks) < min(n, T):
        picks.add(int(rng.integers(0, T)))
    return np.array(sorted(picks), dtype=np.int64)
