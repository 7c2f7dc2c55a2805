"""The mixed serving step at full size: 32 layers x {qkv 4096->6144, o 4096->4096, gate_up
4096->28672, down 14336->4096}, 1024 tokens (4 prefill requests of 192 tokens, then 256 decode
tokens, one request each), tenants drawn Zipf(1.1) over 1000 registered adapters of ranks
[8, 16, 64][id mod 3] (alpha = 2r), admitted into 128 slots in three rank classes (8, 16, 64).

All 128 pools and weights live on the GPU (about 30 GB). The oracle checks every linear on a
block of token rows x output columns: rows in every 128-token tile and the first token of every
slot in use, 96 random columns plus the first and last; the W and B rows it needs are
regenerated on the host from the counter-based input generator, so the full matrices never
leave the device."""
import numpy as np
import pytest

import oracle
import synth
from tests.harness import assert_close, errors

pytestmark = pytest.mark.gpu

N_LAYERS = 32
R_MAX = 64
N_SLOTS = 128


class _Sub:
    """An adapter restricted to sampled output rows of B (for the oracle)."""

    def __init__(self, ad, cols):
        self.A, self.B, self.rank, self.alpha, self.rslora = ad.A, ad.B[cols], ad.rank, ad.alpha, ad.rslora


def _rows_to_check(plan, rng):
    """One or two rows per 128-token tile, both ends of every prefill segment, and the first
    token of every slot in use."""
    T = plan["T"]
    ts = plan["token_slots"][:, 0]
    rows = {0, T - 1, 191, 192, 383, 384, 575, 576, 767, 768}
    for t0 in range(0, T, 128):
        rows.update(int(t) for t in rng.integers(t0, min(T, t0 + 128), size=2))
    for s in np.unique(ts[ts >= 0]):
        rows.add(int(np.argmax(ts == s)))
    return np.array(sorted(rows), dtype=np.int64)


def test_mixed_serving_step_full_size(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora

    plan = synth.mixed_step_plan()
    seed, T = plan["seed"], plan["T"]
    slot_of, rank_of = plan["slot_of"], plan["rank_of"]
    classes = plan["classes"]
    assert len(slot_of) <= N_SLOTS and sum(n for n, _ in classes) == N_SLOTS
    adapters_by_slot = {s: a for a, s in slot_of.items()}

    free, total = torch.cuda.mem_get_info()
    if free < 40 * 2 ** 30:
        pytest.skip(f"needs about 35 GB of free device memory, {free / 2 ** 30:.0f} GB free")

    meta = layer.StepMeta(T, 1, R_MAX)
    token_slots = torch.from_numpy(plan["token_slots"]).cuda()
    rng = np.random.default_rng(7)
    rows = _rows_to_check(plan, rng)

    linears = []          # (layer, module, K, D, pool, W_dev, x_dev, y_dev)
    for l in range(N_LAYERS):
        for m, (name, K, D, _) in enumerate(synth.MIXED_MODULES):
            pool = layer.AdapterPool(N_SLOTS, R_MAX, K, D, classes=classes)
            for s, a in adapters_by_slot.items():
                ad = synth.mixed_adapter(seed, l, m, a, K, D)
                assert ad.rank == rank_of[a]
                mlora.mlora_load_adapter(pool.handle, s, ad.A, ad.B, ad.rank, ad.alpha, ad.rslora)
            W = layer.bf16_from_bits(synth.mixed_weight_rows(seed, l, m, K, 0, D), "cuda")
            x = layer.bf16_from_bits(synth.mixed_x(seed, l, m, T, K), "cuda")
            y = torch.empty((T, D), dtype=torch.float32, device="cuda")
            linears.append((l, m, K, D, pool, W, x, y))
    for lin in linears:
        lin[4].sync()

    # one step: metadata once, then all 128 linears
    meta.build(token_slots, None, linears[0][4])
    for (l, m, K, D, pool, W, x, y) in linears:
        layer.linear(pool, meta, x, W, y)
    torch.cuda.synchronize()
    meta.status()
    m_dev = meta.read()
    assert m_dev == oracle.meta(plan["token_slots"], N_SLOTS)

    worst = (0.0, 0.0)
    for (l, m, K, D, pool, W, x, y) in linears:
        cols = np.unique(np.concatenate([[0, D - 1], rng.choice(D, size=96, replace=False)]))
        W_sub = np.stack([synth.mixed_weight_rows(seed, l, m, K, int(o), 1)[0] for o in cols])
        subs = {s: _Sub(synth.mixed_adapter(seed, l, m, a, K, D), cols) for s, a in adapters_by_slot.items()}
        x_host = synth.mixed_x(seed, l, m, T, K)
        ref = oracle.linear(x_host, W_sub, plan["token_slots"], subs, N_SLOTS, rows=rows)
        got = y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
        rel, mx = assert_close(got, ref, f"layer {l} {synth.MIXED_MODULES[m][0]}")
        worst = (max(worst[0], rel), max(worst[1], mx))
    print(f"mixed step: worst rel Frobenius {worst[0]:.2e}, worst max-abs {worst[1]:.2e}")
    for lin in linears:
        lin[4].close()
    meta.close()
