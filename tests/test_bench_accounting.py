"""The bench's algorithmic byte counts (the roofline numerators), recomputed by hand from the
workload's slot table for the small-batch path and for a wide output, on CPU."""
import numpy as np

import bench
import synth


def _distinct(slots):
    return sorted(set(int(s) for s in slots[slots >= 0]))


def test_small_batch_path_bytes():
    wl = synth.decode(T=64, n_adapters=12)
    got = bench.algorithmic_bytes(wl, num_sms=152)
    d = _distinct(wl.token_slots)
    R = (wl.r_max + 7) // 8 * 8
    rows = int(np.any(wl.token_slots >= 0, axis=1).sum())
    pairs = int((wl.token_slots >= 0).sum())
    base = exp = 0
    for l in wl.linears:
        base += l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4          # W, x, y
        base += len(d) * R * l.K * 2 + wl.T * len(d) * R * 4              # A rows, v of every token
        rb = sum((l.adapters[s].rank + 7) // 8 * 8 for s in d)
        exp += rb * l.D * 2 + rows * l.D * 8 + pairs * R * 4              # B rows, y RMW, v reads
    assert got["base_gemm"] == base and got["expand"] == exp and got["shrink"] == 0
    assert got["base_flops"] == sum(2 * wl.T * l.K * l.D for l in wl.linears)


def test_wide_output_leaves_the_small_batch_path():
    wl = synth.logits(T=32, vocab=152 * 128 + 8, hidden=256)             # one column block too many
    got = bench.algorithmic_bytes(wl, num_sms=152)
    l = wl.linears[0]
    d = _distinct(wl.token_slots)
    R = (wl.r_max + 7) // 8 * 8
    rows = int(np.any(wl.token_slots >= 0, axis=1).sum())
    pairs = int((wl.token_slots >= 0).sum())
    assert got["base_gemm"] == l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4
    ra = sum(l.adapters[s].rank for s in d)
    rb = sum((l.adapters[s].rank + 7) // 8 * 8 for s in d)
    assert got["shrink"] == ra * l.K * 2 + rows * l.K * 2 + pairs * R * 4
    assert got["expand"] == rb * l.D * 2 + rows * l.D * 8 + pairs * R * 4
    # one block narrower: back on the small-batch path (A rows and v in the GEMM's count)
    narrow = synth.logits(T=32, vocab=152 * 128, hidden=256)
    assert bench.algorithmic_bytes(narrow, num_sms=152)["shrink"] == 0
