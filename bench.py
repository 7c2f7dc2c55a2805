"""Benchmark of the multi-LoRA batched linear layer on GB300.

Workload (default): the decode batch of the pages' shapes -- 256 tokens at hidden 4096
through four q/k/v/o-shaped 4096 -> 4096 bf16 linears, each with its own pool of 100
resident rank-16 adapters (alpha 32); per-token slot uniform over the 100 with 10 % of
tokens on the sentinel -1. One step = build the slot metadata once, then the four
linears (base GEMM + shrink + expand each). Metric: tokens per second through the step.

Output: one JSON line (rank 0). Kernel durations for the roofline come from a second
pass of the same K steps with per-kernel CUDA events (the library's trace), so that the
events do not slow the headline timing. L2 is flushed (256 MiB write) before every timed
step, outside the timed events.

--impl reference times the fp64 CPU oracle (the only reference this subject has) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-linear tokens/s (1×GB300) + % of HBM / bf16 tensor roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


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
def make_workload(name: str):
    import synth
    if name == "decode":
        return synth.decode()
    if name == "logits":
        return synth.logits()
    if name == "compose":
        return synth.compose()
    if name == "tiny":
        return synth.tiny()
    if name == "prefill":
        return synth.prefill()
    if name == "mixed":
        return synth.mixed()
    raise SystemExit(f"unknown workload {name}")


def workload_config(wl, name: str) -> dict:
    lin = wl.linears
    return {
        "workload": f"{name}: T={wl.T} tokens, J={wl.J}, linears "
                    + (", ".join(f"{l.name} {l.K}->{l.D}" for l in lin) if len(lin) <= 8 else
                       f"{len(lin) // 4} layers x (" + ", ".join(f"{l.name.split('.')[-1]} {l.K}->{l.D}" for l in lin[:4]) + ")")
                    + f", {wl.n_slots} slots r_max={wl.r_max}",
        "tokens_per_step": wl.T,
        "linears": len(lin),
        "slots": wl.n_slots,
        "r_max": wl.r_max,
        "slots_per_token": wl.J,
        "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
    }


def algorithmic_bytes(wl, num_sms: int = 152) -> dict:
    """Bytes each kernel kind must move per step (unique data, each counted once), by path.

    Small batches (T <= 256 and every output's 128-column blocks within one wave of the SMs: one
    split-K tensor-core kernel computes the base product and the shrink of every active slot): base_gemm = W + x + y write (fp32) + A rows of the active slots
    (R rows each, the pool's padded rank) + v write (T x active slots x R, fp32); expand = B rows
    of the active slots at the true rank padded to 8 + read and write of y rows with an active
    slot + v reads of the active pairs.
    Larger batches with rank width 64, 128-token tiles of at most four slots (tensor-core path):
    shrink = A rows (64 per slot) + x rows of those tiles + the scaled bf16 v tiles written;
    base_gemm = W + x + y + those v tiles read again + B rows (64 columns per slot). Pairs in
    tiles with more slots, and every pair of other larger batches: shrink = A rows at the true
    rank + x rows of active tokens + v partial writes; expand = B rows + y read-modify-write +
    v reads.
    Flops: 2*T*K*D per linear for the base product."""
    slots = wl.token_slots
    active = slots >= 0
    R = (wl.r_max + 7) // 8 * 8
    small = wl.T <= 256 and all((l.D + 127) // 128 <= num_sms for l in wl.linears)
    tensor_core = wl.T > 256 and R == 64
    fused = np.zeros_like(active)
    tile_slots = []                                   # distinct slots of each fused 128-token tile
    if tensor_core:
        for t0 in range(0, wl.T, 128):
            d = set(int(s) for s in slots[t0:t0 + 128][active[t0:t0 + 128]])
            if len(d) <= 4:
                fused[t0:t0 + 128] = active[t0:t0 + 128]
                tile_slots.append((min(128, wl.T - t0), d))
    rest = active & ~fused
    act_rows = int(np.any(rest, axis=1).sum())
    pairs = int(rest.sum())
    distinct = sorted(set(int(s) for s in slots[rest]))
    tc_slots = sorted(set().union(*(d for _, d in tile_slots))) if tile_slots else []
    tc_rows = sum(rows for rows, d in tile_slots if d)
    tc_vtile = sum(rows * len(d) * 64 * 2 for rows, d in tile_slots)
    out = {"base_gemm": 0, "shrink": 0, "expand": 0, "base_flops": 0, "meta": wl.T * wl.J * 4 * 6}
    for l in wl.linears:
        out["base_gemm"] += l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4
        out["base_flops"] += 2 * wl.T * l.K * l.D
        ra = sum(l.adapters[s].rank for s in distinct)
        rb = sum((l.adapters[s].rank + 7) // 8 * 8 for s in distinct)
        if small:
            out["base_gemm"] += len(distinct) * R * l.K * 2 + wl.T * len(distinct) * R * 4
            out["expand"] += rb * l.D * 2 + act_rows * l.D * 8 + pairs * R * 4
            continue
        if tc_slots:
            out["shrink"] += len(tc_slots) * 64 * l.K * 2 + tc_rows * l.K * 2 + tc_vtile
            out["base_gemm"] += tc_vtile + len(tc_slots) * 64 * l.D * 2
        if pairs:
            out["shrink"] += ra * l.K * 2 + act_rows * l.K * 2 + pairs * R * 4
            out["expand"] += rb * l.D * 2 + act_rows * l.D * 8 + pairs * R * 4
    return out


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
    growing number of token rows until about budget_s of CPU work. Returns tokens/s, rows, threads."""
    import oracle
    threads = oracle.default_threads()
    T = wl.T
    # a step whose tensors are generated on demand (the mixed step): time its first layer and
    # scale to all layers (every layer has the same shapes and adapter set)
    scale = 1.0
    if any(l.W is None for l in wl.linears):
        first = wl.linears[:len(synth_modules())]
        scale = len(wl.linears) / len(first)
        if getattr(wl, "_first_layer", None) is None:     # generated once per workload object
            wl._first_layer = type(wl)(wl.name, wl.seed, wl.T, wl.J, wl.n_slots, wl.r_max, wl.token_slots,
                                       wl.scales, {l.x_id: synth_x(wl, l) for l in first},
                                       [synth_materialize(wl, l) for l in first])
        wl = wl._first_layer
    cap = T if max_rows is None else min(T, max_rows)
    rows_n = min(cap, max(1, threads))
    spent, tokens = 0.0, 0
    rng = np.random.default_rng(0)
    while True:
        rows = np.sort(rng.choice(T, size=rows_n, replace=False))
        t0 = time.perf_counter()
        for l in wl.linears:
            oracle.linear(wl.xs[l.x_id], l.W, wl.token_slots, l.adapters, wl.n_slots, scales=wl.scales,
                          rows=rows, threads=threads)
        real = time.perf_counter() - t0
        spent += real
        tokens = rows_n
        last = real * scale
        if rows_n >= cap or spent + real * 2.5 > budget_s:
            break
        rows_n = min(cap, rows_n * 2)
    return tokens / last, tokens, threads, last


def synth_modules():
    import synth
    return synth.MIXED_MODULES


def synth_x(wl, lin):
    import synth
    return synth.materialize_x(wl, lin)


def synth_materialize(wl, lin):
    import synth
    return synth.materialize_linear(wl, lin)


def sample_note(wl, rows, seconds=None) -> str:
    lazy = any(l.W is None for l in wl.linears)
    what = (f"{rows} of {wl.T} token rows through the first {len(synth_modules())} of {len(wl.linears)} "
            f"linears, time scaled to all of them" if lazy else
            f"{rows} of {wl.T} token rows through all {len(wl.linears)} linears")
    return what + (f" ({seconds:.1f} s)" if seconds is not None else " per step")


# ------------------------------------------------------------------------------ reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = make_workload(args.workload)
    step_budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    rows = None
    times = []
    for i in range(args.warmup + args.steps):
        tps, rows, threads, dt = oracle_sample(wl, budget_s=step_budget, max_rows=rows)
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
                         "sample": sample_note(wl, rows)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ our arm
# Sources each recorded kernel is built from; a traffic record holds only while they are unchanged.
KERNEL_SOURCES = {
    ("decode", "base_gemm"): ("gemm_tc.cu", "ptx.cuh", "internal.h"),
    ("decode", "expand"): ("expand_vfull.cu", "expand_vfull.cuh", "ptx.cuh", "internal.h"),
    ("prefill", "base_gemm"): ("gemm_pair.cu", "ptx.cuh", "internal.h"),
    ("prefill", "shrink"): ("sgmv_tc.cu", "lora_kernels.cu", "ptx.cuh", "internal.h"),
    ("logits", "expand"): ("lora_kernels.cu", "ptx.cuh", "internal.h"),
    ("logits", "base_gemm"): ("gemm_pair.cu", "ptx.cuh", "internal.h"),
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


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from rank_adapter_gemm_token_gb300 import mlora
    from tests.harness import DeviceWorkload

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local)) if "device_id" in \
            dist.init_process_group.__code__.co_varnames else dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    __graft_entry__.build()

    wl = make_workload(args.workload)
    dw = DeviceWorkload(wl, device=device)
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

    # The step (metadata build + every linear) is captured once into a CUDA graph and replayed:
    # the same kernels with the same arguments, without per-call host work.
    run_step = lambda: dw.run(stream)  # noqa: E731
    graph = None
    if not args.no_graph:
        cap = torch.cuda.Stream(device)
        with torch.cuda.stream(cap):
            dw.run()                      # first use on the capture stream, outside the capture
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            dw.run()
        torch.cuda.synchronize(device)
        run_step = graph.replay
        for _ in range(args.warmup):
            flush.zero_()
            run_step()
        barrier()

    # ---- headline: K timed steps, L2 flushed before each, no tracing
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = mlora.mlora_launch_count()
    barrier()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    launches = mlora.mlora_launch_count() - launches0 if graph is None else kernels_per_step * args.steps
    clock_info = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms, value = aggregate_over_ranks(float(np.mean(step_ms)), wl.T)

    # ---- per-kernel durations: the same K steps again with the library's event trace
    trace_steps = min(args.steps, 100)
    mlora.mlora_trace_enable(int(kernels_per_step) * trace_steps + 64)
    for i in range(trace_steps):
        flush.zero_()
        dw.run(stream)
    barrier()
    trace = mlora.mlora_trace_read()
    mlora.mlora_trace_disable()

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
    for i in range(args.steps):
        flush.zero_()
        e_start.record(stream)
        e2e_run()
        e_end.record(stream)
        e_end.synchronize()
        e2e_ms.append(e_start.elapsed_time(e_end))
    _, e2e_value = aggregate_over_ranks(float(np.mean(e2e_ms)), wl.T)
    torch.cuda.synchronize(device)
    dw.meta.status()

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    algo = algorithmic_bytes(wl, torch.cuda.get_device_properties(device).multi_processor_count)
    kinds = {k: v for k, v in trace.items() if v[0] > 0}
    dom = max(kinds, key=lambda k: kinds[k][1])
    n_launch, tot_ms = kinds[dom]
    avg_s = tot_ms / n_launch / 1000.0
    launches_per_step = n_launch / trace_steps
    if dom == "base_gemm":
        flops = algo["base_flops"] / launches_per_step
        byts = algo["base_gemm"] / launches_per_step
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        bound = "tensor" if flops / byts > ridge else "hbm"
    else:
        byts = algo.get(dom, 0) / launches_per_step
        flops, bound = 0, "hbm"
    if bound == "tensor":
        achieved, peak, unit = flops / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = byts / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
    roofline = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)"
                if peak_src == "measured" else "fallback",
                "traffic": recorded_traffic(dom, args.workload),
                "algorithmic_bytes_per_launch": byts, "avg_launch_us": avg_s * 1e6}
    per_kernel = {}
    for k, (n, t) in kinds.items():
        per = n / trace_steps
        entry = {"launches_per_step": per, "avg_us": 1000.0 * t / n, "share": t / sum(v[1] for v in kinds.values())}
        if k in algo and algo[k] > 0:
            entry["achieved_GBps"] = algo[k] / per / (t / n / 1000.0) / 1e9
            entry["frac_hbm"] = entry["achieved_GBps"] / peaks["hbm_gbs"]
        if k == "base_gemm":
            entry["achieved_TFLOPs"] = algo["base_flops"] / per / (t / n / 1000.0) / 1e12
            entry["frac_bf16"] = entry["achieved_TFLOPs"] / peaks["bf16_tflops"]
        per_kernel[k] = entry
    # the whole step against its own bound: the slower of (all algorithmic bytes / HBM peak) and
    # (all flops / bf16 peak), over the measured step time
    step_bytes = sum(v for k, v in algo.items() if k not in ("base_flops",))
    bound_s = max(step_bytes / (peaks["hbm_gbs"] * 1e9), algo["base_flops"] / (peaks["bf16_tflops"] * 1e12))
    step_roofline = {"bound_us": bound_s * 1e6, "frac": bound_s / (ms / 1000.0),
                     "bytes_per_step": step_bytes, "flops_per_step": algo["base_flops"]}

    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        tps, rows, threads, dt = oracle_sample(wl, budget_s=args.cpu_budget)
        cpu = {"value": tps, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": sample_note(wl, rows, dt)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Philox4x64-10 + Box-Muller, bf16-rounded)",
        "config": dict(workload_config(wl, args.workload), parallelism=f"replicas x{ws}" if ws > 1 else "single GPU"),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "clocks": clock_info,
        "kernels": per_kernel,
        "step_roofline": step_roofline,
        "wall_s_timed_region": wall,
        "kernel_timing": f"second pass of {trace_steps} steps with per-kernel CUDA events on the launch stream",
        "step_launch": "CUDA graph replay of the captured step" if graph is not None else "direct calls",
    }
    print(json.dumps(line), flush=True)
    dw.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mlora", choices=["mlora", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "compose", "prefill", "tiny", "mixed", "logits"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="call the library directly for every step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
