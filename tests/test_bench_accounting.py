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


def test_tensor_core_path_bytes():
    # 3 requests of 192 tokens plus 64 tokens on five other slots: tiles 0-3 have <= 4 slots
    # (fused: SGMV shrink, expand as extra K blocks), tile 4 has more (left to the other kernels)
    wl = synth.prefill(n_requests=3, seg_len=192, hidden=128, mlp=256)
    tail = np.arange(64, dtype=np.int32) % 5 + 3
    wl.token_slots = np.concatenate([wl.token_slots[:, 0], tail]).reshape(-1, 1)
    wl.T = wl.token_slots.shape[0]
    for lin in wl.linears:
        for s in range(3, 8):
            lin.adapters[s] = lin.adapters[s % 3]
    got = bench.algorithmic_bytes(wl, num_sms=152)
    slots = wl.token_slots[:, 0]
    fused_tiles = [(min(128, wl.T - t0), set(slots[t0:t0 + 128].tolist())) for t0 in range(0, wl.T, 128)
                   if len(set(slots[t0:t0 + 128].tolist())) <= 4]
    assert len(fused_tiles) == 5 - 1
    tc_slots = sorted(set().union(*(d for _, d in fused_tiles)))
    tc_rows = sum(r for r, _ in fused_tiles)
    vtile = sum(r * len(d) * 64 * 2 for r, d in fused_tiles)
    rest = np.zeros(wl.T, bool)
    rest[512:] = True                                              # tile 4 (tokens 512 .. 639)
    d = sorted(set(slots[rest].tolist()))
    shrink = base = exp = 0
    for l in wl.linears:
        base += l.D * l.K * 2 + wl.T * l.K * 2 + wl.T * l.D * 4 + vtile + len(tc_slots) * 64 * l.D * 2
        shrink += len(tc_slots) * 64 * l.K * 2 + tc_rows * l.K * 2 + vtile
        shrink += sum(l.adapters[s].rank for s in d) * l.K * 2 + int(rest.sum()) * l.K * 2 + int(rest.sum()) * 64 * 4
        exp += sum((l.adapters[s].rank + 7) // 8 * 8 for s in d) * l.D * 2 + int(rest.sum()) * l.D * 8 \
            + int(rest.sum()) * 64 * 4
    assert (got["base_gemm"], got["shrink"], got["expand"]) == (base, shrink, exp)
