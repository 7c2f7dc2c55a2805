"""Benchmark of the multi-LoRA batched linear layer on GB300.

Workload (default): the mixed serving step -- a Llama-style stack of 32 layers x {qkv
4096 -> 6144, o 4096 -> 4096, gate_up 4096 -> 28672, down 14336 -> 4096} in bf16, 1024 tokens
(4 prefill segments of 192 tokens, one adapter each, then 256 decode tokens, one request
each), tenants Zipf(1.1) over 1000 registered adapters of ranks 8/16/64 admitted into 128 GPU
slots. One step = build the slot metadata once, then every linear (base GEMM + shrink +
expand). Metric: tokens per second through the step. Other workloads (decode, prefill,
compose, logits, tiny, and the embedding lookup with LoRA on the mixed step's tokens) are
behind --workload.

Output: one JSON line (rank 0). Kernel durations for the roofline come from a second pass of
the same steps with per-kernel CUDA events (the library's trace), so that the events do not
slow the headline timing. L2 is flushed (256 MiB write) before every timed step, outside the
timed events. The line also carries the step split into its phases (the prefill tokens alone
and the decode tokens alone, each against its own bound), the adapter load rate (host to
device, per slot) and the end-to-end rate through the C ABI with host buffers.

--impl reference times the fp64 CPU oracle (the only reference this subject has) on a
bounded sample of the same workload on the host cores.

--gpus N (N > 1) runs one replica of the workload per GPU (tokens are independent rows; no
collective on the data path): launched under torchrun it takes WORLD_SIZE ranks, started
directly it starts torchrun itself.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-linear tokens/s (1×GB300) + % of HBM / bf16 tensor roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOADS = ("mixed", "decode", "compose", "prefill", "tiny", "logits", "embedding")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def tensor_peak_for(peaks: dict, peak_src: str, clock_info) -> tuple:
    """The bf16 denominator for this run: the sustained figure (a seconds-long matmul loop under
    the power cap) when the power cap throttled the SM clock during the timed steps, so that the
    kernels ran in that regime inside a long step; else the burst figure (kernels timed alone).
    Returns (peaks with bf16_tflops set accordingly, a note naming the choice)."""
    reasons = (clock_info or {}).get("reasons") or []
    if "sw_power_cap" in reasons and "bf16_tflops_sustained" in peaks:
        chosen = dict(peaks, bf16_tflops=peaks["bf16_tflops_sustained"])
        which = "bf16 sustained: sw_power_cap active during the timed steps"
    else:
        chosen, which = dict(peaks), "bf16 burst"
    note = f"measured (MEASURED_PEAKS.json; {which})" if peak_src == "measured" else f"fallback ({which})"
    return chosen, note


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def headline_fields(ms_local: float, tokens_per_rank: int) -> dict:
    """The line's whole-job fields from this rank's mean step time: the slowest rank's time and
    the tokens of all ranks over it (one replica per rank)."""
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms, value = aggregate_over_ranks(ms_local, tokens_per_rank)
    return {"value": value, "n_gpus": ws, "ms_per_step": ms, "scaling": "weak",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}


def aggregate_over_ranks(ms_local: float, tokens_per_rank: int) -> tuple:
    """Whole-job timing: the slowest rank's ms per step and tokens/s over all ranks (each rank
    runs its own replica of the workload, so the work per rank is fixed: weak scaling)."""
    import torch
    import torch.distributed as dist
    ws = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms = float(ms_local)
    if ws > 1:
        dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, ws * tokens_per_rank / (ms / 1000.0)


# ------------------------------------------------------------------------------ workload
def make_workload(name: str, layers: int = 32):
    import synth
    if name == "mixed":
        return synth.mixed(n_layers=layers)
    if name == "embedding":
        return synth.embedding_step()
    return {"decode": synth.decode, "logits": synth.logits, "compose": synth.compose, "tiny": synth.tiny,
            "prefill": synth.prefill}[name]()


def workload_config(wl, name: str) -> dict:
    if name == "embedding":
        return {
            "workload": f"embedding: {wl.T} tokens of the mixed step through a {wl.vocab} x {wl.dim} table with LoRA, "
                        f"J={wl.J}, {wl.n_slots} slots in rank classes {wl.classes}",
            "tokens_per_step": wl.T, "vocab": wl.vocab, "dim": wl.dim, "slots": wl.n_slots, "r_max": wl.r_max,
            "slots_per_token": wl.J,
            "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
        }
    lin = wl.linears
    if len(lin) <= 8:
        what = ", ".join(f"{l.name} {l.K}->{l.D}" for l in lin)
    else:
        what = f"{len(lin) // 4} layers x 4 linears (" + ", ".join(
            f"{l.name.split('.')[-1]} {l.K}->{l.D}" for l in lin[:4]) + ")"
    phases = "".join(f", {b - a} {n}" for n, a, b in getattr(wl, "phases", []))
    return {
        "workload": f"{name}: {wl.T} tokens{phases}, J={wl.J}, linears {what}, {wl.n_slots} slots r_max={wl.r_max}",
        "tokens_per_step": wl.T,
        "linears": len(lin),
        "slots": wl.n_slots,
        "r_max": wl.r_max,
        "slots_per_token": wl.J,
        "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
    }


def sub_workload(wl, r0: int, r1: int):
    """The same linears and adapters over token rows [r0, r1) (a phase of the step)."""
    import copy
    sub = copy.copy(wl)
    sub.T = r1 - r0
    sub.token_slots = wl.token_slots[r0:r1]
    sub.scales = None if wl.scales is None else wl.scales[r0:r1]
    sub.xs = {k: v[r0:r1] for k, v in wl.xs.items()}
    sub.phases = []
    return sub


FUSE_MAX_K = 8192     # the library's CTA-pair GEMM computes the shrink itself up to this K


def layer_path(wl, lin, num_sms: int = 152) -> str:
    """Which kernels the library runs for this linear: 'small' (T <= 256, one rank width, output
    column blocks within one wave: split-K GEMM with the shrink folded in, then a separate expand),
    'fused' (two or more 128-token tiles and K <= 8192: the CTA-pair GEMM computes the shrink as
    sub-tiles of its schedule and the expand as extra K blocks) or 'tc' (the separate tensor-core
    shrink, then the expand inside the base GEMM as extra K blocks)."""
    classes = getattr(wl, "classes", None)
    if wl.T <= 256 and not classes and (lin.D + 127) // 128 <= num_sms:
        return "small"
    if wl.T > 128 and lin.K <= FUSE_MAX_K:
        return "fused"
    return "tc"


def algorithmic(wl, num_sms: int = 152) -> dict:
    """Bytes and flops the method must move and do per step (each tensor counted once, adapters
    at their true rank), attributed to the kernel that moves them.

    Per linear: W [D, K] + x [T, K] (bf16) and the fp32 output y [T, D]; the A rows and B rows of
    every adapter that at least one token uses, at its true rank; v (fp32, one value per active
    pair and rank row) written by the shrink and read by the expand. Where the expand runs as its
    own kernel after the GEMM ('small' path) it also reads and writes y on the rows that have an
    active slot; where it runs inside the base GEMM ('tc' path) y is written once.
    Flops: 2 T K D for the base product, 2 r K per active pair for the shrink, 2 r D per active
    pair for the expand.
    Attribution: 'small': base_gemm = W + x + y + A rows + v write, expand = B rows + y
    read-modify-write + v read. 'tc': shrink = A rows + x rows of the tokens with an active slot
    + v write, base_gemm = W + x + y + B rows + v read. 'fused': all of it to base_gemm (W + x + y
    + A rows + B rows + v written and read), with the shrink's flops."""
    slots = wl.token_slots
    active = slots >= 0
    rows = int(np.any(active, axis=1).sum())
    distinct = sorted(set(int(s) for s in slots[active]))
    out = {k: 0 for k in ("meta", "base_gemm", "shrink", "expand")}
    flops = {k: 0 for k in ("base_gemm", "shrink", "expand")}
    out["meta"] = wl.T * wl.J * 4 * 6
    for l in wl.linears:
        ranks = {s: l.adapters[s].rank for s in distinct}
        sum_r = sum(ranks.values())
        pair_r = int(sum(ranks[int(s)] for s in slots[active]))
        v = pair_r * 4
        base = l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4
        a_rows, b_rows = sum_r * l.K * 2, sum_r * l.D * 2
        f_base, f_shrink, f_expand = 2 * wl.T * l.K * l.D, 2 * pair_r * l.K, 2 * pair_r * l.D
        path = layer_path(wl, l, num_sms)
        if path == "small":
            out["base_gemm"] += base + a_rows + v
            out["expand"] += b_rows + rows * l.D * 8 + v
            flops["base_gemm"] += f_base + f_shrink
            flops["expand"] += f_expand
        elif path == "fused":
            out["base_gemm"] += base + a_rows + b_rows + 2 * v
            flops["base_gemm"] += f_base + f_shrink + f_expand
        else:
            out["shrink"] += a_rows + rows * l.K * 2 + v
            out["base_gemm"] += base + b_rows + v
            flops["shrink"] += f_shrink
            flops["base_gemm"] += f_base + f_expand
    out["flops"] = flops
    return out


def algorithmic_embedding(wl) -> dict:
    """Bytes and flops of the embedding lookup with LoRA per step: each token's table row (bf16)
    and its fp32 output row, the ids, the token's A column of every active pair (r bf16 values),
    B of every adapter in use once (at its true rank); flops 2 r D per active pair. The metadata
    build: 24 bytes per pair."""
    slots = wl.token_slots
    active = slots >= 0
    distinct = sorted(set(int(s) for s in slots[active]))
    pair_r = int(sum(wl.adapters[int(s)].rank for s in slots[active]))
    emb = wl.T * wl.dim * (2 + 4) + wl.T * 4 + pair_r * 2 + sum(wl.adapters[s].rank for s in distinct) * wl.dim * 2
    return {"meta": wl.T * wl.J * 4 * 6, "embedding": emb, "flops": {"embedding": 2 * pair_r * wl.dim}}


def roofline_of(byts: float, flops: float, seconds: float, peaks: dict) -> dict:
    """A kernel (or step) against the roofline: bound by whichever of bytes / HBM peak and
    flops / bf16 peak takes longer."""
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    bound = "tensor" if flops / tc > byts / hbm else "hbm"
    if bound == "tensor":
        achieved, peak, unit = flops / seconds / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = byts / seconds / 1e9, peaks["hbm_gbs"], "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "bound_us": max(flops / tc, byts / hbm) * 1e6, "hbm_frac": byts / hbm / seconds,
            "tensor_frac": flops / tc / seconds}


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples the SM clock, its maximum and the clock-event (throttle) reasons through NVML
    (ctypes, read-only queries) from a thread every ~0.5 ms while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        import threading
        self.samples, self.error, self.h = [], None, None
        self._stop = threading.Event()
        self._thread = None
        try:
            import ctypes
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            uuid = None
            try:
                import torch
                u = getattr(torch.cuda.get_device_properties(cuda_index), "uuid", None)
                if u is not None:
                    uuid = "GPU-" + str(u)
            except Exception:
                pass
            ok = uuid is not None and self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            if not ok and self.nvml.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.h = h
        except OSError as e:
            self.error = str(e)

    def _run(self):
        import ctypes
        mhz, mx, mask = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if (self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0 and
                    self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 and
                    get_reasons(self.h, ctypes.byref(mask)) == 0):
                self.samples.append((mhz.value, mx.value, mask.value))
            time.sleep(0.0005)

    def start(self):
        import threading
        if self.h is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self) -> dict:
        if self._thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"NVML unavailable: {self.error}"]}
        self._stop.set()
        self._thread.join()
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for _, _, m in self.samples:
            for bit, name in self.REASONS.items():
                if m & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([s[0] for s in self.samples])),
                "sm_max_mhz": float(max(s[1] for s in self.samples)), "samples": len(self.samples),
                "reasons": sorted(reasons), "source": "NVML, sampled during the timed steps"}


# ------------------------------------------------------------------------------ oracle timing
def oracle_sample(wl, budget_s: float = 12.0, max_rows: int | None = None):
    """Times the fp64 oracle on a bounded sample of the workload: all linears of the step for a
    growing number of token rows until about budget_s of CPU work. A step whose tensors are
    generated on demand (the mixed step) is timed on its first layer and the time scaled to all
    layers (every layer has the same shapes and adapter set). Returns (tokens/s, rows, threads,
    seconds per step for those rows, extrapolated)."""
    import oracle
    import synth
    threads = oracle.default_threads()
    T = wl.T
    scale = 1.0
    lazy = any(l.W is None for l in wl.linears)
    if lazy:
        first = wl.linears[:len(synth.MIXED_MODULES)]
        scale = len(wl.linears) / len(first)
        if getattr(wl, "_first_layer", None) is None:     # generated once per workload object
            import copy
            fl = copy.copy(wl)
            fl.xs = {l.x_id: synth.materialize_x(wl, l) for l in first}
            fl.linears = [synth.materialize_linear(wl, l) for l in first]
            wl._first_layer = fl
        wl = wl._first_layer
    cap = T if max_rows is None else min(T, max_rows)
    rows_n = min(cap, max(1, threads))
    spent = 0.0
    rng = np.random.default_rng(0)
    while True:
        rows = np.sort(rng.choice(T, size=rows_n, replace=False))
        t0 = time.perf_counter()
        for l in wl.linears:
            oracle.linear(wl.xs[l.x_id], l.W, wl.token_slots, l.adapters, wl.n_slots, scales=wl.scales,
                          rows=rows, threads=threads)
        real = time.perf_counter() - t0
        spent += real
        last = real * scale
        if rows_n >= cap or spent + real * 2.5 > budget_s:
            break
        rows_n = min(cap, rows_n * 2)
    return rows_n / last, rows_n, threads, last, lazy


def oracle_sample_embedding(wl, budget_s: float = 12.0, max_rows: int | None = None):
    """The embedding oracle on a growing sample of token rows until about budget_s of CPU work;
    returns (tokens/s, rows, threads, seconds for those rows, extrapolated=False)."""
    import oracle
    cap = wl.T if max_rows is None else min(wl.T, max_rows)
    rows_n, spent = min(cap, 16), 0.0
    rng = np.random.default_rng(0)
    while True:
        rows = np.sort(rng.choice(wl.T, size=rows_n, replace=False))
        t0 = time.perf_counter()
        oracle.embedding(wl.ids, wl.E, wl.token_slots, wl.adapters, wl.n_slots, scales=wl.scales, rows=rows)
        real = time.perf_counter() - t0
        spent += real
        if rows_n >= cap or spent + real * 2.5 > budget_s:
            break
        rows_n = min(cap, rows_n * 2)
    return rows_n / real, rows_n, 1, real, False


def sample_note(wl, rows, seconds=None, lazy=False) -> str:
    if not hasattr(wl, "linears"):
        return f"{rows} of {wl.T} token rows through the embedding oracle" + (
            f" ({seconds:.2f} s per step)" if seconds is not None else " per step")
    import synth
    what = (f"{rows} of {wl.T} token rows through the first {len(synth.MIXED_MODULES)} of {len(wl.linears)} "
            f"linears, time extrapolated to all of them" if lazy else
            f"{rows} of {wl.T} token rows through all {len(wl.linears)} linears")
    return what + (f" ({seconds:.1f} s per step, extrapolated)" if seconds is not None and lazy else
                   f" ({seconds:.2f} s per step)" if seconds is not None else " per step")


# ------------------------------------------------------------------------------ reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = make_workload(args.workload, args.layers)
    step_budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    rows = None
    times = []
    lazy = False
    threads = 1
    sampler = oracle_sample_embedding if args.workload == "embedding" else oracle_sample
    for i in range(args.warmup + args.steps):
        _, rows, threads, dt, lazy = sampler(wl, budget_s=step_budget, max_rows=rows)
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * float(np.mean(times))
    value = rows / (ms / 1000.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Philox4x64-10 + Box-Muller, bf16-rounded)",
        "config": workload_config(wl, args.workload),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample_note(wl, rows, lazy=lazy), "extrapolated": lazy},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ our arm
# Sources each recorded kernel is built from; a traffic record holds only while they are unchanged.
KERNEL_SOURCES = {
    ("mixed", "base_gemm"): ("gemm_pair.cu", "ptx.cuh", "internal.h"),
    ("mixed", "shrink"): ("shrink_tc.cu", "ptx.cuh", "internal.h"),
    ("decode", "base_gemm"): ("gemm_tc.cu", "ptx.cuh", "internal.h"),
    ("decode", "expand"): ("expand_vfull.cu", "expand_vfull.cuh", "ptx.cuh", "internal.h"),
    ("prefill", "base_gemm"): ("gemm_pair.cu", "ptx.cuh", "internal.h"),
    ("prefill", "shrink"): ("shrink_tc.cu", "ptx.cuh", "internal.h"),
    ("logits", "base_gemm"): ("gemm_pair.cu", "ptx.cuh", "internal.h"),
    ("embedding", "embedding"): ("embedding.cu", "ptx.cuh", "internal.h"),
}


def kernel_hash(files=None) -> str:
    """sha256 prefix over the named kernel sources (all of csrc/ when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rank_adapter_gemm_token_gb300", "csrc")
    for n in sorted(files if files is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.json), or None when
    missing or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or (workload, kind) not in KERNEL_SOURCES:
        return None
    try:
        rec = json.load(open(path))
    except ValueError:
        return None
    r = rec.get(workload, {}).get(kind)
    if not r or r.get("kernel_hash") != kernel_hash(KERNEL_SOURCES[(workload, kind)]):
        return None
    return r.get("dram_bytes_per_launch")


def time_graph(run, steps: int, warmup: int, stream, flush, device, barrier):
    """Captures run() once into a CUDA graph and times `steps` replays (L2 flushed before each)
    with CUDA events on `stream`; returns (ms per replay, graph)."""
    import torch
    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        run()                                  # first use on the capture stream, outside the capture
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        run()
    torch.cuda.synchronize(device)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
    barrier()
    return float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)])), graph


def time_adapter_loads(dw, n_slots: int = 16):
    """Host-to-device adapter load rate: re-loads up to n_slots resident adapters of the largest
    linear from pinned host buffers (the pinning done beforehand) and times the queued copies until
    the pool's loads are complete (wall clock)."""
    import torch
    import synth
    from rank_adapter_gemm_token_gb300 import mlora
    dl = max(dw.linears, key=lambda d: d.lin.K + d.lin.D)
    lin = dl.lin
    staged = []
    for s, ad in sorted(lin.adapters.items())[:n_slots]:
        if isinstance(ad, synth.LazyAdapter):
            ad = ad.materialize(lin.K, lin.D)
        a = torch.from_numpy(np.ascontiguousarray(ad.A).view(np.int16)).pin_memory()
        b = torch.from_numpy(np.ascontiguousarray(ad.B).view(np.int16)).pin_memory()
        staged.append((s, a, b, ad))
    torch.cuda.synchronize()
    nbytes = sum(a.numel() * 2 + b.numel() * 2 for _, a, b, _ in staged)
    t0 = time.perf_counter()
    for s, a, b, ad in staged:
        mlora.mlora_load_adapter(dl.pool.handle, s, a.data_ptr(), b.data_ptr(), ad.rank, ad.alpha, ad.rslora)
    dl.pool.sync()
    dt = time.perf_counter() - t0
    return {"linear": f"{lin.name} {lin.K}->{lin.D}", "slots": len(staged), "bytes": nbytes,
            "ms_per_slot": 1000.0 * dt / max(1, len(staged)), "h2d_GBps": nbytes / dt / 1e9,
            "how": "mlora_load_adapter from pinned host memory on the pool's copy stream, wall clock until "
                   "mlora_pool_sync returns (slot A zeroing, A copy, B copy into a staging buffer, "
                   "scatter kernel into the slot's B columns, slot factor)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from rank_adapter_gemm_token_gb300 import mlora
    from tests.harness import DeviceWorkload

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        if "device_id" in dist.init_process_group.__code__.co_varnames:
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    __graft_entry__.build()

    t_setup = time.perf_counter()
    wl = make_workload(args.workload, args.layers)
    dw = DeviceWorkload(wl, device=device)
    torch.cuda.synchronize(device)
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        flush.zero_()
        dw.run(stream)
    dw.meta.status()
    barrier()
    l0 = mlora.mlora_launch_count()
    dw.run(stream)
    kernels_per_step = mlora.mlora_launch_count() - l0
    barrier()

    # ---- headline: K timed steps, L2 flushed before each, no tracing. The step (metadata build +
    # every linear) is captured once into a CUDA graph and replayed: the same kernels with the same
    # arguments, without per-call host work.
    clocks = ClockSampler(local)
    clocks.start()
    wall0 = time.perf_counter()
    if args.no_graph:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            dw.run(stream)
            ends[i].record(stream)
        barrier()
        ms_local = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))
    else:
        ms_local, _ = time_graph(lambda: dw.run(), args.steps, args.warmup, stream, flush, device, barrier)
    wall = time.perf_counter() - wall0
    clock_info = clocks.stop()
    launches = kernels_per_step * args.steps
    head = headline_fields(ms_local, wl.T)

    # ---- per-kernel durations: the same steps again with the library's event trace
    trace_steps = min(args.steps, 20)
    mlora.mlora_trace_enable(int(kernels_per_step) * trace_steps + 64)
    for _ in range(trace_steps):
        flush.zero_()
        dw.run(stream)
    barrier()
    trace = mlora.mlora_trace_read()
    mlora.mlora_trace_disable()

    # ---- phases: the prefill tokens alone and the decode tokens alone, through the same linears
    burst_peaks, peak_src = load_peaks()
    peaks, peak_note = tensor_peak_for(burst_peaks, peak_src, clock_info)
    num_sms = torch.cuda.get_device_properties(device).multi_processor_count
    phases = {}
    for name, r0, r1 in getattr(wl, "phases", []):
        sub = dw.sub_rows(r0, r1)
        p_ms, _ = time_graph(lambda: sub.run(), max(3, min(args.steps, 20)), 3, stream, flush, device, barrier)
        sw = sub_workload(wl, r0, r1)
        pa = algorithmic(sw, num_sms)
        rf = roofline_of(sum(v for k, v in pa.items() if k != "flops"), sum(pa["flops"].values()), p_ms / 1000.0, peaks)
        phases[name] = {"tokens": r1 - r0, "us": p_ms * 1000.0, "bound": rf["bound"], "bound_us": rf["bound_us"],
                        "frac": rf["bound_us"] / (p_ms * 1000.0), "hbm_frac": rf["hbm_frac"],
                        "tensor_frac": rf["tensor_frac"]}
        sub.close()

    # ---- end to end: pinned host inputs in, step, result out, every step
    xs_host = {k: v.cpu().pin_memory() for k, v in dw.x.items()}
    slots_host = dw.token_slots.cpu().pin_memory()
    scales_host = None if dw.scales is None else dw.scales.cpu().pin_memory()
    ys_host = [torch.empty(dl.y.shape, dtype=dl.y.dtype).pin_memory() for dl in dw.linears]
    h2d = sum(v.numel() * v.element_size() for v in xs_host.values()) + slots_host.numel() * 4 + \
        (0 if scales_host is None else scales_host.numel() * 4)
    d2h = sum(y.numel() * y.element_size() for y in ys_host)
    # The step as a user would pipeline it through the public API: the inputs go up on a copy
    # stream, each linear waits only for its own input, and each output goes down on a second
    # copy stream while the next linear computes. Captured once as a graph (with the flag
    # --no-graph, issued directly each step).
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def e2e_step(s):
        up.wait_stream(s)
        down.wait_stream(s)
        ev_x = {}
        with torch.cuda.stream(up):
            dw.token_slots.copy_(slots_host, non_blocking=True)
            if scales_host is not None:
                dw.scales.copy_(scales_host, non_blocking=True)
            ev_meta = torch.cuda.Event()
            ev_meta.record(up)
            for k, v in xs_host.items():
                dw.x[k].copy_(v, non_blocking=True)
                ev_x[k] = torch.cuda.Event()
                ev_x[k].record(up)
        s.wait_event(ev_meta)
        dw.build_meta(s)
        for dl, yh in zip(dw.linears, ys_host):
            s.wait_event(ev_x[dl.lin.x_id])
            dw.layer.linear(dl.pool, dw.meta, dw.x[dl.lin.x_id], dl.W, dl.y, s)
            ev_y = torch.cuda.Event()
            ev_y.record(s)
            down.wait_event(ev_y)
            with torch.cuda.stream(down):
                yh.copy_(dl.y, non_blocking=True)
        s.wait_stream(up)
        s.wait_stream(down)

    e2e_run = lambda: e2e_step(stream)  # noqa: E731
    if not args.no_graph:
        cap = torch.cuda.Stream(device)
        e2e_step(cap)                    # first use of the streams and events, outside the capture
        torch.cuda.synchronize(device)
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=cap):
            e2e_step(cap)
        torch.cuda.synchronize(device)
        e2e_run = e2e_graph.replay
    for _ in range(args.warmup):
        e2e_run()
    torch.cuda.synchronize(device)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(max(3, min(args.steps, 20))):
        flush.zero_()
        e_start.record(stream)
        e2e_run()
        e_end.record(stream)
        e_end.synchronize()
        e2e_ms.append(e_start.elapsed_time(e_end))
    _, e2e_value = aggregate_over_ranks(float(np.mean(e2e_ms)), wl.T)
    torch.cuda.synchronize(device)
    dw.meta.status()

    load_rate = time_adapter_loads(dw)

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        dw.close()
        return 0

    # ---- roofline of the dominant kernel
    algo = algorithmic(wl, num_sms)
    kinds = {k: v for k, v in trace.items() if v[0] > 0}
    dom = max(kinds, key=lambda k: kinds[k][1])
    n_launch, tot_ms = kinds[dom]
    avg_s = tot_ms / n_launch / 1000.0
    per_step = n_launch / trace_steps
    rf = roofline_of(algo.get(dom, 0) / per_step, algo["flops"].get(dom, 0) / per_step, avg_s, peaks)
    roofline = {"kernel": dom, "bound": rf["bound"], "achieved": rf["achieved"], "peak": rf["peak"],
                "unit": rf["unit"], "frac": rf["frac"], "peak_source": peak_note,
                "frac_of_burst_peak": rf["achieved"] / (burst_peaks["bf16_tflops"] if rf["bound"] == "tensor"
                                                         else burst_peaks["hbm_gbs"]),
                "traffic": recorded_traffic(dom, args.workload),
                "algorithmic_bytes_per_launch": algo.get(dom, 0) / per_step,
                "algorithmic_flops_per_launch": algo["flops"].get(dom, 0) / per_step,
                "avg_launch_us": avg_s * 1e6}
    per_kernel = {}
    total_traced = sum(v[1] for v in kinds.values())
    for k, (n, t) in kinds.items():
        per = n / trace_steps
        entry = {"launches_per_step": per, "avg_us": 1000.0 * t / n, "share": t / total_traced}
        kb, kf = algo.get(k, 0) / per, algo["flops"].get(k, 0) / per
        if kb > 0:
            entry["achieved_GBps"] = kb / (t / n / 1000.0) / 1e9
            entry["frac_hbm"] = entry["achieved_GBps"] / peaks["hbm_gbs"]
        if kf > 0:
            entry["achieved_TFLOPs"] = kf / (t / n / 1000.0) / 1e12
            entry["frac_bf16"] = entry["achieved_TFLOPs"] / peaks["bf16_tflops"]
        per_kernel[k] = entry
    # the whole step against its own bound: the slower of (all algorithmic bytes / HBM peak) and
    # (all flops / bf16 peak), over the measured step time; and each fraction alone
    step_bytes = sum(v for k, v in algo.items() if k != "flops")
    step_flops = sum(algo["flops"].values())
    srf = roofline_of(step_bytes, step_flops, ms_local / 1000.0, peaks)
    step_roofline = {"bound": srf["bound"], "bound_us": srf["bound_us"], "frac": srf["bound_us"] / (ms_local * 1000.0),
                     "hbm_frac": srf["hbm_frac"], "tensor_frac": srf["tensor_frac"],
                     "bytes_per_step": step_bytes, "flops_per_step": step_flops}

    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        tps, rows, threads, dt, lazy = oracle_sample(wl, budget_s=args.cpu_budget)
        cpu = {"value": tps, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": sample_note(wl, rows, dt, lazy), "extrapolated": lazy}

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": head["n_gpus"], "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": head["scaling"], "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox4x64-10 + Box-Muller, bf16-rounded)",
        "config": dict(workload_config(wl, args.workload), parallelism=head["parallelism"]),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clock_info,
        "kernels": per_kernel,
        "step_roofline": step_roofline,
        "phases": phases,
        "adapter_load": load_rate,
        "setup_s": setup_s,
        "wall_s_timed_region": wall,
        "kernel_timing": f"second pass of {trace_steps} steps with per-kernel CUDA events on the launch stream",
        "step_launch": "direct calls" if args.no_graph else "CUDA graph replay of the captured step",
    }
    print(json.dumps(line), flush=True)
    dw.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_embedding(args):
    """The embedding lookup with LoRA on the mixed step's tokens: one step = the metadata build and
    one mlora_embedding call, captured as a graph and replayed; the same JSON line as the linear
    workloads (roofline of the dominant kernel, step roofline, e2e with host buffers, oracle
    baseline on a row sample)."""
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from rank_adapter_gemm_token_gb300 import layer, mlora

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    __graft_entry__.build()

    t_setup = time.perf_counter()
    wl = make_workload("embedding")
    pool = layer.EmbeddingPool(wl.vocab, wl.dim, wl.classes)
    for s_, ad in wl.adapters.items():
        pool.load(s_, ad.A, ad.B, ad.rank, ad.alpha, ad.rslora)
    pool.sync()
    E = layer.bf16_from_bits(wl.E, device)
    ids = torch.from_numpy(wl.ids.astype(np.int32)).to(device)
    slots = torch.from_numpy(np.ascontiguousarray(wl.token_slots.astype(np.int32))).to(device)
    meta = layer.StepMeta(wl.T, wl.J, wl.r_max)
    y = torch.empty((wl.T, wl.dim), dtype=torch.float32, device=device)
    torch.cuda.synchronize(device)
    setup_s = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    def step(s=None):
        meta.build(slots, None, pool, s)
        layer.embedding(pool, meta, ids, E, y, s)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        flush.zero_()
        step(stream)
    meta.status()
    barrier()
    l0 = mlora.mlora_launch_count()
    step(stream)
    kernels_per_step = mlora.mlora_launch_count() - l0
    barrier()

    clocks = ClockSampler(local)
    clocks.start()
    wall0 = time.perf_counter()
    ms_local, _ = time_graph(lambda: step(), args.steps, args.warmup, stream, flush, device, barrier)
    wall = time.perf_counter() - wall0
    clock_info = clocks.stop()
    head = headline_fields(ms_local, wl.T)

    trace_steps = min(args.steps, 20)
    mlora.mlora_trace_enable(int(kernels_per_step) * trace_steps + 64)
    for _ in range(trace_steps):
        flush.zero_()
        step(stream)
    barrier()
    trace = mlora.mlora_trace_read()
    mlora.mlora_trace_disable()

    # end to end: ids and token slots up from pinned host memory, the step, y down
    ids_h, slots_h = ids.cpu().pin_memory(), slots.cpu().pin_memory()
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()

    def e2e_step():
        ids.copy_(ids_h, non_blocking=True)
        slots.copy_(slots_h, non_blocking=True)
        step()
        y_h.copy_(y, non_blocking=True)

    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        e2e_step()
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        e2e_step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(device)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(max(3, min(args.steps, 20))):
        flush.zero_()
        e_start.record(stream)
        graph.replay()
        e_end.record(stream)
        e_end.synchronize()
        e2e_ms.append(e_start.elapsed_time(e_end))
    _, e2e_value = aggregate_over_ranks(float(np.mean(e2e_ms)), wl.T)
    meta.status()
    h2d, d2h = ids_h.numel() * 4 + slots_h.numel() * 4, y_h.numel() * 4

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    burst_peaks, peak_src = load_peaks()
    peaks, peak_note = tensor_peak_for(burst_peaks, peak_src, clock_info)
    algo = algorithmic_embedding(wl)
    kinds = {k: v for k, v in trace.items() if v[0] > 0}
    dom = max(kinds, key=lambda k: kinds[k][1])
    n_launch, tot_ms = kinds[dom]
    avg_s = tot_ms / n_launch / 1000.0
    per_step = n_launch / trace_steps
    rf = roofline_of(algo.get(dom, 0) / per_step, algo["flops"].get(dom, 0) / per_step, avg_s, peaks)
    roofline = {"kernel": dom, "bound": rf["bound"], "achieved": rf["achieved"], "peak": rf["peak"],
                "unit": rf["unit"], "frac": rf["frac"], "peak_source": peak_note,
                "traffic": recorded_traffic(dom, "embedding"),
                "algorithmic_bytes_per_launch": algo.get(dom, 0) / per_step,
                "algorithmic_flops_per_launch": algo["flops"].get(dom, 0) / per_step,
                "avg_launch_us": avg_s * 1e6}
    total_traced = sum(v[1] for v in kinds.values())
    per_kernel = {k: {"launches_per_step": n / trace_steps, "avg_us": 1000.0 * t / n, "share": t / total_traced}
                  for k, (n, t) in kinds.items()}
    step_bytes = sum(v for k, v in algo.items() if k != "flops")
    srf = roofline_of(step_bytes, sum(algo["flops"].values()), ms_local / 1000.0, peaks)
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        tps, rows, threads, dt, _ = oracle_sample_embedding(wl, budget_s=args.cpu_budget)
        cpu = {"value": tps, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample_note(wl, rows, dt),
               "extrapolated": False}
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": head["n_gpus"], "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": head["scaling"], "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox4x64-10 + Box-Muller, bf16-rounded)",
        "config": dict(workload_config(wl, "embedding"), parallelism=head["parallelism"]),
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(kernels_per_step * args.steps), "clocks": clock_info, "kernels": per_kernel,
        "step_roofline": {"bound": srf["bound"], "bound_us": srf["bound_us"],
                          "frac": srf["bound_us"] / (ms_local * 1000.0), "hbm_frac": srf["hbm_frac"],
                          "bytes_per_step": step_bytes},
        "setup_s": setup_s, "wall_s_timed_region": wall,
        "kernel_timing": f"second pass of {trace_steps} steps with per-kernel CUDA events on the launch stream",
        "step_launch": "CUDA graph replay of the captured step",
    }
    print(json.dumps(line), flush=True)
    pool.close()
    meta.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mlora", choices=["mlora", "reference"])
    ap.add_argument("--workload", default="mixed", choices=WORKLOADS)
    ap.add_argument("--layers", type=int, default=32, help="layers of the mixed step (a smaller case for captures)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="call the library directly for every step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start them under torchrun (rendezvous on the loopback address)
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__),
               *(sys.argv[1:] if argv is None else argv)]
        return subprocess.call(cmd)
    ws = dist_env()[0]
    if ws != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={ws}: launch one rank per GPU")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "embedding":
        return run_embedding(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
