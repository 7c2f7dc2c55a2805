"""The bench's algorithmic byte and flop counts (the roofline numerators), recomputed by hand from
the workload's slot table, on CPU: only the method's bytes (adapters at their true rank, one v
value per active pair and rank row), attributed to the kernel that moves them."""
import numpy as np

import bench
import synth


def _distinct(slots):
    return sorted(set(int(s) for s in slots[slots >= 0]))


def _pair_ranks(wl, lin):
    return sum(lin.adapters[int(s)].rank for s in wl.token_slots[wl.token_slots >= 0])


def test_small_batch_path_counts_only_the_methods_v():
    wl = synth.decode(T=64, n_adapters=12)
    got = bench.algorithmic(wl, num_sms=152)
    d = _distinct(wl.token_slots)
    rows = int(np.any(wl.token_slots >= 0, axis=1).sum())
    base = exp = fb = fe = 0
    for l in wl.linears:
        sr = sum(l.adapters[s].rank for s in d)
        pr = _pair_ranks(wl, l)
        base += l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4 + sr * l.K * 2 + pr * 4
        exp += sr * l.D * 2 + rows * l.D * 8 + pr * 4
        fb += 2 * wl.T * l.K * l.D + 2 * pr * l.K
        fe += 2 * pr * l.D
    assert (got["base_gemm"], got["expand"], got["shrink"]) == (base, exp, 0)
    assert got["flops"] == {"base_gemm": fb, "shrink": 0, "expand": fe}
    # not the dense table of every token against every active slot
    assert got["base_gemm"] < sum(l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4 for l in wl.linears) + \
        len(wl.linears) * (len(d) * 16 * 4096 * 2 + wl.T * len(d) * 16 * 4)


def test_wide_output_takes_the_tensor_core_path():
    wl = synth.logits(T=32, vocab=152 * 128 + 8, hidden=256)             # one column block too many
    got = bench.algorithmic(wl, num_sms=152)
    l = wl.linears[0]
    d = _distinct(wl.token_slots)
    rows = int(np.any(wl.token_slots >= 0, axis=1).sum())
    sr = sum(l.adapters[s].rank for s in d)
    pr = _pair_ranks(wl, l)
    assert got["shrink"] == sr * l.K * 2 + rows * l.K * 2 + pr * 4
    assert got["base_gemm"] == l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4 + sr * l.D * 2 + pr * 4
    assert got["expand"] == 0
    assert got["flops"]["base_gemm"] == 2 * wl.T * l.K * l.D + 2 * pr * l.D
    narrow = synth.logits(T=32, vocab=152 * 128, hidden=256)
    assert bench.layer_path(narrow, narrow.linears[0], 152) == "small"


def test_large_batch_counts_each_adapter_once():
    # K <= 8192 and two or more 128-token tiles: the pair GEMM computes the shrink itself, so every
    # byte and flop of the side path is the GEMM's
    wl = synth.prefill(n_requests=3, seg_len=192, hidden=128, mlp=256)
    got = bench.algorithmic(wl, num_sms=152)
    base = fl = 0
    for l in wl.linears:
        assert bench.layer_path(wl, l, 152) == "fused"
        sr = sum(l.adapters[s].rank for s in range(3))
        pr = _pair_ranks(wl, l)
        base += l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4 + sr * l.K * 2 + sr * l.D * 2 + 2 * pr * 4
        fl += 2 * wl.T * l.K * l.D + 2 * pr * l.K + 2 * pr * l.D
    assert (got["shrink"], got["base_gemm"], got["expand"]) == (0, base, 0)
    assert got["flops"]["base_gemm"] == fl


def test_long_k_keeps_the_separate_shrink():
    wl = synth.prefill(n_requests=3, seg_len=192, hidden=128, mlp=9000)   # the down projection: K > 8192
    got = bench.algorithmic(wl, num_sms=152)
    shrink = 0
    for l in wl.linears:
        if l.K <= bench.FUSE_MAX_K:
            continue
        assert bench.layer_path(wl, l, 152) == "tc"
        sr = sum(l.adapters[s].rank for s in range(3))
        shrink += sr * l.K * 2 + wl.T * l.K * 2 + _pair_ranks(wl, l) * 4
    assert got["shrink"] == shrink > 0


def test_roofline_picks_the_slower_bound():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0}
    r = bench.roofline_of(byts=1e9, flops=1e12, seconds=0.02, peaks=peaks)   # 1 ms of bytes, 10 ms of flops
    assert r["bound"] == "tensor" and abs(r["bound_us"] - 10000.0) < 1e-6 and abs(r["frac"] - 0.5) < 1e-12
    r = bench.roofline_of(byts=1e10, flops=1e12, seconds=0.02, peaks=peaks)  # 10 ms of bytes, 10 ms of flops
    assert r["bound"] == "hbm" and abs(r["hbm_frac"] - 0.5) < 1e-12


def test_phase_rows_cover_the_mixed_step():
    plan = synth.mixed(n_layers=1)
    names = [p[0] for p in plan.phases]
    assert names == ["prefill", "decode"]
    assert plan.phases[0][1] == 0 and plan.phases[-1][2] == plan.T
    assert plan.phases[0][2] == plan.phases[1][1] == 768
    sub = bench.sub_workload(plan, 768, plan.T)
    assert sub.T == 256 and sub.token_slots.shape == (256, 1)


def test_tensor_peak_follows_the_power_cap():
    # the sustained bf16 figure only when the power cap throttled the timed steps; HBM unchanged
    peaks = {"hbm_gbs": 6698.2, "bf16_tflops": 1883.1, "bf16_tflops_sustained": 1710.1}
    capped, note = bench.tensor_peak_for(peaks, "measured", {"reasons": ["sw_power_cap"]})
    assert capped["bf16_tflops"] == 1710.1 and capped["hbm_gbs"] == 6698.2 and "sustained" in note
    for clocks in ({"reasons": []}, {"reasons": ["hw_slowdown"]}, None, {}):
        free, note = bench.tensor_peak_for(peaks, "measured", clocks)
        assert free["bf16_tflops"] == 1883.1 and "burst" in note
    assert peaks["bf16_tflops"] == 1883.1                       # the caller's dict is left alone
    rf = bench.roofline_of(1e6, 1.7e12, 1e-3, capped)           # 1.7 PFLOP/s of work for 1 ms
    assert rf["bound"] == "tensor" and abs(rf["frac"] - 1700.0 / 1710.1) < 1e-9
