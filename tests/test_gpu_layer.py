"""The full layer on the GPU against the fp64 oracle, through the C ABI.

Tolerances: relative Frobenius error <= 5e-3 and max-abs error <= 3e-2 per linear output,
also applied to the LoRA delta alone (y - base) for the relative error. Rows whose slots
are all -1 must equal the base product bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests.conftest import read_golden
from tests.harness import DeviceWorkload, assert_close, errors, oracle_rows, sample_rows, tile_rows

pytestmark = pytest.mark.gpu


def _sentinel_run(dw, dl):
    """The same layer call with every slot set to -1 (same shapes, pool and grid)."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    meta = layer.StepMeta(dw.wl.T, dw.wl.J, dw.wl.r_max)
    meta.build(torch.full_like(dw.token_slots, -1), None, dl.pool)
    out = layer.linear(dl.pool, meta, dw.x[dl.lin.x_id], dl.W).cpu().numpy()
    meta.close()
    return out


def _check_linear(wl, dw, dl, rows=None, check_delta=True):
    from rank_adapter_gemm_token_gb300 import layer
    y = dl.y.cpu().numpy()
    ref = oracle_rows(wl, dl.lin, rows=rows)
    ysel = y if rows is None else y[rows]
    assert_close(ysel, ref, f"{wl.name}/{dl.lin.name}")
    base_dev = _sentinel_run(dw, dl)
    bsel = base_dev if rows is None else base_dev[rows]
    # rows with no active slot equal the base product of the same call exactly
    slots = wl.token_slots if rows is None else wl.token_slots[rows]
    idle = np.all(slots < 0, axis=1)
    assert np.array_equal(ysel[idle], bsel[idle]), "sentinel rows differ from the base product"
    # ... and the standalone base GEMM up to fp32 summation order
    gemm = layer.base_gemm(dw.x[dl.lin.x_id], dl.W).cpu().numpy()
    gsel = gemm if rows is None else gemm[rows]
    rel, _ = errors(bsel, gsel.astype(np.float64))
    assert rel < 1e-5, f"base product differs from the standalone GEMM: {rel:.2e}"
    if check_delta and (~idle).any():
        base_ref = oracle.linear(wl.xs[dl.lin.x_id], dl.lin.W, np.full((wl.T, 1), -1), {}, wl.n_slots, rows=rows)
        rel, _ = errors(ysel[~idle] - bsel[~idle], ref[~idle] - base_ref[~idle])
        assert rel <= 5e-3, f"LoRA delta alone: rel Frobenius {rel:.3e}"


def test_hand_example_is_bit_exact(cuda_device):
    """The hand-worked two-slot example, zero-padded to K = D = 8: every value is exact in fp32,
    so the GPU must reproduce the hand-computed outputs exactly."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    g = {k: v for k, v in read_golden("hand_two_slot_rslora.txt") if k != "slot"}
    slot_lines = [v for k, v in read_golden("hand_two_slot_rslora.txt") if k == "slot"]
    T, K0, D0, J = (int(g[k][0]) for k in ("T", "K", "D", "J"))
    K = D = 8
    f = lambda k: np.array([float(v) for v in g[k]], dtype=np.float32)  # noqa: E731
    bits = lambda a: (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    x = np.zeros((T, K), np.float32); x[:, :K0] = f("x").reshape(T, K0)
    W = np.zeros((D, K), np.float32); W[:D0, :K0] = f("W").reshape(D0, K0)
    pool = layer.AdapterPool(int(g["n_slots"][0]), 4, K, D)
    for sl in slot_lines:
        s = int(sl[0]); kv = dict(zip(sl[1::2], sl[2::2])); r = int(kv["rank"])
        A = np.zeros((r, K), np.float32); A[:, :K0] = f(f"A{s}").reshape(r, K0)
        B = np.zeros((D, r), np.float32); B[:D0] = f(f"B{s}").reshape(D0, r)
        pool.load(s, bits(A), bits(B), r, float(kv["alpha"]), bool(int(kv["rslora"])))
    pool.sync()
    meta = layer.StepMeta(T, J, 4)
    ts = torch.tensor(np.array([int(v) for v in g["token_slots"]], np.int32).reshape(T, J), device="cuda")
    sc = torch.tensor(f("scales").reshape(T, J), device="cuda")
    meta.build(ts, sc, pool)
    y = layer.linear(pool, meta, layer.bf16_from_bits(bits(x), "cuda"), layer.bf16_from_bits(bits(W), "cuda"))
    meta.status()
    expect = np.zeros((T, D)); expect[:, :D0] = f("y").reshape(T, D0)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), expect)


def test_tiny_config(cuda_device):
    wl = synth.tiny()
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])
    dw.close()


@pytest.mark.parametrize("T,K,D,S,R,J,seed", [(300, 200, 520, 7, 16, 2, 0), (129, 264, 136, 3, 64, 1, 1),
                                              (77, 64, 8, 12, 8, 3, 2), (513, 1024, 384, 40, 24, 2, 3)])
def test_ragged_multi_slot_cases(cuda_device, T, K, D, S, R, J, seed):
    """Several tiles with ragged tails, mixed ranks below r_max, rsLoRA, J slots with sentinels."""
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(rng.integers(1, 3 * r)), rslora=bool(s % 3 == 0))
    slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    slots[::5, :] = -1
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("ragged", seed, T, J, S, R, slots, scales, {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])
    dw.close()


def test_decode_config_full_size(cuda_device):
    # every token row of every linear
    wl = synth.decode()
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    for dl in dw.linears:
        _check_linear(wl, dw, dl)
    dw.close()


@pytest.mark.parametrize("path", [1, 2])
def test_decode_shapes_on_both_paths(cuda_device, path):
    """The decode configuration's shapes forced onto the small-batch path (1) and onto the
    tensor-core side path (2): both against the oracle on sampled rows."""
    from rank_adapter_gemm_token_gb300 import mlora
    wl = synth.decode()
    wl.linears = wl.linears[:2]
    mlora.mlora_set_path(path)
    try:
        dw = DeviceWorkload(wl)
        dw.run()
        dw.meta.status()
        rows = sample_rows(wl, 40)
        for dl in dw.linears:
            _check_linear(wl, dw, dl, rows=rows)
        dw.close()
    finally:
        mlora.mlora_set_path(0)


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("T,K,D,S,R,J,seed", [(250, 200, 4100, 30, 16, 1, 80), (33, 264, 600, 9, 32, 2, 81),
                                              (1, 72, 136, 3, 8, 1, 82), (176, 512, 1000, 12, 64, 3, 83),
                                              (256, 4096, 4096, 100, 16, 1, 84)])
def test_small_batch_gemm_forms(cuda_device, skinny_form, form, T, K, D, S, R, J, seed):
    """The small-batch path with each form of its GEMM (1: split-K CTA pairs; 2: token groups with
    W and x rows shared by multicast) and the shrink folded in: ragged token counts (groups with
    padding rows), a partial last output block, several slots per token, rank up to R; against
    the oracle, and bit-identical over repeated steps."""
    from rank_adapter_gemm_token_gb300 import mlora
    skinny_form(form)
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(rng.integers(1, 3 * r)), rslora=bool(s % 3 == 0))
    slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    slots[::7, :] = -1
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("forms", seed, T, J, S, R, slots, scales, {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])
    mlora.mlora_set_path(1)
    try:
        dw = DeviceWorkload(wl)
        dw.run()
        dw.meta.status()
        first = dw.linears[0].y.cpu().numpy()
        dw.run()
        dw.meta.status()
        assert np.array_equal(dw.linears[0].y.cpu().numpy(), first), "the small-batch path is not deterministic"
        rows = None if T * D <= 300_000 else sample_rows(wl, 40)
        _check_linear(wl, dw, dw.linears[0], rows=rows)
        dw.close()
    finally:
        mlora.mlora_set_path(0)


def test_compose_config_full_size(cuda_device):
    wl = synth.compose()
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])                     # every token row
    # RFC 51940, Testing: the fused k-slot pass equals running one slot at a time and accumulating.
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    dl = dw.linears[0]
    fused = dl.y.clone()
    acc = layer.base_gemm(dw.x[0], dl.W)
    meta1 = layer.StepMeta(wl.T, 1, wl.r_max)
    for j in range(wl.J):
        meta1.build(dw.token_slots[:, j].contiguous().view(wl.T, 1), dw.scales[:, j].contiguous(), dl.pool)
        layer.linear(dl.pool, meta1, dw.x[0], dl.W, dl.y)
        acc += dl.y - layer.base_gemm(dw.x[0], dl.W)
    rel, mx = errors(fused.cpu().numpy(), acc.cpu().numpy().astype(np.float64))
    assert rel < 1e-5 and mx < 1e-4, (rel, mx)
    dw.close()


def test_prefill_config_full_size(cuda_device):
    # rows in every one of the 32 tiles (first, last and two more) and of every slot
    wl = synth.prefill()
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    rows = tile_rows(wl, per_tile=2)
    assert len(set(int(r) // 128 for r in rows)) == (wl.T + 127) // 128
    for dl in dw.linears:
        _check_linear(wl, dw, dl, rows=rows)
    dw.close()


@pytest.mark.parametrize("T,J", [(256, 2), (1024, 2), (256, 1), (1, 2), (7, 1)])
def test_lm_head_router_mixture(cuda_device, T, J):
    """The side path on the LM head (hidden 4096 -> a 32000-entry vocabulary) with router-weighted
    mixtures: two adapters per token with per-token gate weights ("[RFC] Per-request activation
    of multiple LoRA adapters", related work: router-driven mixtures; "[vLLM] LoRA",
    add_lora_logits: the LM head takes the same shrink and expand). A 32000-wide output has
    more 128-column blocks than SMs, so both batch sizes take the tiled GEMM with the separate
    shrink and expand of a 32-wide pool (T = 1 and 7: a single 128-row tile, one-CTA GEMM); J = 1
    takes the slot-sorted expand, J = 2 the per-token one."""
    wl = synth.logits(T=T, vocab=32000, J=J)
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0], rows=sample_rows(wl, 12))
    dw.close()


def test_zero_scale_and_linearity_on_gpu(cuda_device):
    import torch
    wl = synth.compose(T=64)
    dw = DeviceWorkload(wl)
    outs = {}
    for s in (0.0, 1.0, 0.5):
        dw.scales = torch.full((wl.T, wl.J), s, dtype=torch.float32, device="cuda")
        dw.run()
        outs[s] = dw.linears[0].y.cpu().numpy().astype(np.float64)
    base = _sentinel_run(dw, dw.linears[0])
    assert np.array_equal(outs[0.0], base)                  # zero scale adds exact zeros
    rel, _ = errors(outs[0.5] - base, 0.5 * (outs[1.0] - base))
    assert rel < 1e-6
    dw.close()


def test_reload_slot_after_use(cuda_device):
    """Write-after-read: reloading a slot that a queued linear still reads must not change that
    linear's result, and the next linear sees the new adapter."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    wl = synth.tiny(T=64)
    dw = DeviceWorkload(wl)
    dl = dw.linears[0]
    y_first = torch.empty_like(dl.y)
    dw.build_meta()
    layer.linear(dl.pool, dw.meta, dw.x[0], dl.W, y_first)
    new = synth.Adapter(A=synth.normal_bf16(99, 1, (8, wl.linears[0].K), 0.02),
                        B=synth.normal_bf16(99, 2, (wl.linears[0].D, 8), 0.02), rank=8, alpha=8.0)
    dl.pool.load(1, new.A, new.B, new.rank, new.alpha, new.rslora)
    layer.linear(dl.pool, dw.meta, dw.x[0], dl.W, dl.y)
    torch.cuda.synchronize()
    rows = np.arange(wl.T)
    assert_close(y_first.cpu().numpy(), oracle_rows(wl, wl.linears[0], rows=rows), "before reload")
    wl.linears[0].adapters[1] = new
    assert_close(dl.y.cpu().numpy(), oracle_rows(wl, wl.linears[0], rows=rows), "after reload")
    dw.close()


def test_load_errors(cuda_device):
    from rank_adapter_gemm_token_gb300 import layer, mlora
    pool = layer.AdapterPool(4, 16, 64, 64)
    A = np.zeros((32, 64), np.uint16)
    B = np.zeros((64, 32), np.uint16)
    with pytest.raises(mlora.MloraError) as e:
        pool.load(0, A, B, 32, 64.0)
    assert e.value.status == mlora.MLORA_ERR_RANK_TOO_LARGE and "32" in str(e.value) and "16" in str(e.value)
    with pytest.raises(mlora.MloraError) as e:
        pool.load(4, A[:8], B[:, :8], 8, 16.0)
    assert e.value.status == mlora.MLORA_ERR_SLOT_RANGE
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_load_adapter(pool.handle, 0, A[:8], np.ascontiguousarray(B[:, :8]), 8, float("nan"), 0)
    assert e.value.status == mlora.MLORA_ERR_RANK_INVALID
    pool.close()


def test_clear_slot_makes_it_empty(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    wl = synth.tiny()
    dw = DeviceWorkload(wl)
    dw.linears[0].pool.clear(2)
    dw.run()
    if (wl.token_slots == 2).any():
        with pytest.raises(mlora.MloraError) as e:
            dw.meta.status()
        assert e.value.status == mlora.MLORA_ERR_BAD_TOKEN_SLOT
    dw.close()


@pytest.mark.parametrize("J,seed,T,K,D,bn", [(1, 5, 700, 320, 392, 0), (2, 6, 700, 320, 392, 0),
                                              (1, 7, 1900, 328, 2504, 0), (2, 8, 1900, 328, 2504, 0),
                                              (1, 9, 1900, 328, 2504, 224), (2, 10, 1500, 200, 1000, 128),
                                              (1, 11, 1500, 200, 1000, 256)])
def test_tensor_core_path_runs_then_random_slots(cuda_device, J, seed, T, K, D, bn):
    """T > 256 with r_max 64: runs of one slot (M-tiles with one or two units) followed by per-token
    random slots (tiles with many units); all on the tensor-core side path (shrink per unit, expand
    inside the base GEMM). Ragged T, K and D; mixed ranks; a second slot per token for J = 2.
    The 1900 x 2504 cases have enough 256 x 256 tiles for the CTA-pair GEMM, an odd number of
    128-row M-tiles (the last pair tile has one) and pairs of M-tiles with different unit lists."""
    rng = np.random.default_rng(seed)
    S, R = 12, 64
    seg_end = 5 * T // 7
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = (8, 16, 64, 40)[s % 4]
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 3 == 0))
    slots = np.full((T, J), -1, dtype=np.int32)
    t = 0
    while t < seg_end:                              # segments of one slot (some of them -1)
        n = int(rng.integers(40, 170))
        slots[t:t + n, 0] = int(rng.integers(-1, S))
        t += n
    slots[seg_end:, 0] = rng.integers(-1, S, size=T - seg_end)
    if J == 2:
        slots[:, 1] = np.where(rng.uniform(size=T) < 0.5, rng.integers(0, S, size=T), -1)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("tc-prefill", seed, T, J, S, R, slots, scales,
                        {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])
    from rank_adapter_gemm_token_gb300 import mlora
    mlora.mlora_set_gemm_tile_n(bn)              # 0: automatic; else the CTA-pair GEMM with this N tile
    try:
        dw = DeviceWorkload(wl)
        dw.run()
        dw.meta.status()
        _check_linear(wl, dw, dw.linears[0])
        dw.close()
    finally:
        mlora.mlora_set_gemm_tile_n(0)


@pytest.mark.parametrize("J,seed,T,ovf", [(1, 50, 700, (4, 5)), (2, 51, 700, (4, 5)), (1, 52, 900, (1, 5)),
                                          (1, 53, 640, (2,)), (2, 54, 1100, (0, 8))])
def test_tiles_with_many_slots(cuda_device, J, seed, T, ovf):
    """T > 256, rank width 64: the tiles listed in ovf draw a slot per token from 40 adapters
    (tens of units per tile), the others use runs of one slot. Covers one and two such tiles,
    adjacent or not, a ragged last tile, and J = 2."""
    rng = np.random.default_rng(seed)
    K, D, S, R = 320, 392, 40, 64
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = (8, 16, 64, 40)[s % 4]
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 3 == 0))
    slots = np.full((T, J), -1, dtype=np.int32)
    for t0 in range(0, T, 128):
        t1 = min(T, t0 + 128)
        if t0 // 128 in ovf:
            slots[t0:t1, 0] = rng.integers(-1, S, size=t1 - t0)
            if J == 2:
                slots[t0:t1, 1] = np.where(rng.uniform(size=t1 - t0) < 0.5, rng.integers(0, S, size=t1 - t0), -1)
        else:
            slots[t0:t0 + 70, 0] = int(rng.integers(0, S))
            slots[t0 + 70:t1, 0] = int(rng.integers(-1, S))
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("many-slots", seed, T, J, S, R, slots, scales,
                        {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])
    dw.close()


@pytest.mark.parametrize("T,J,r,r_max,seed", [(100, 1, 8, 32, 60), (100, 2, 8, 32, 61), (700, 1, 16, 64, 62)])
def test_sliced_adapters_of_a_fused_linear(cuda_device, T, J, r, r_max, seed):
    """Per-slice adapters of a fused qkv-like linear (slices 256 / 64 / 64 wide), loaded with
    mlora_load_adapter_sliced, against the oracle that computes each slice as its own linear.
    T = 100 takes the small-batch path, T = 700 (runs of one slot, rank width 64) the tensor-core
    prefill path."""
    import torch
    from types import SimpleNamespace
    from rank_adapter_gemm_token_gb300 import layer, mlora
    rng = np.random.default_rng(seed)
    K, widths, S = 512, [256, 64, 64], 6
    D = sum(widths)
    W = synth.normal_bf16(seed, 10, (D, K), 0.02)
    x = synth.normal_bf16(seed, 11, (T, K), 1.0)
    sliced = {}
    for s in range(S):
        alpha, rs = float(2 * r), bool(s % 2)
        sliced[s] = [SimpleNamespace(A=synth.normal_bf16(seed, 100 + 10 * s + i, (r, K), 0.02),
                                     B=synth.normal_bf16(seed, 500 + 10 * s + i, (w, r), 0.02),
                                     rank=r, alpha=alpha, rslora=rs) for i, w in enumerate(widths)]
    if T > 256:
        slots = np.repeat(rng.integers(-1, S, size=(T + 127) // 128), 128)[:T].reshape(T, 1).astype(np.int32)
        slots = np.concatenate([slots] * J, axis=1)
    else:
        slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    pool = layer.AdapterPool(S, r_max, K, D)
    for s, parts in sliced.items():
        mlora.mlora_load_adapter_sliced(pool.handle, s, [p.A for p in parts], [p.B for p in parts], r,
                                        parts[0].alpha, parts[0].rslora)
    pool.sync()
    meta = layer.StepMeta(T, J, r_max)
    meta.build(torch.from_numpy(slots).cuda(), torch.from_numpy(scales).cuda(), pool)
    y = layer.linear(pool, meta, layer.bf16_from_bits(x, "cuda"), layer.bf16_from_bits(W, "cuda"))
    meta.status()
    ref = oracle.linear_sliced(x, W, slots, sliced, S, widths, scales=scales)
    assert_close(y.cpu().numpy(), ref, f"sliced T={T} J={J}")
    meta.close()
    pool.close()


def test_sliced_adapter_argument_checks(cuda_device):
    from rank_adapter_gemm_token_gb300 import layer, mlora
    pool = layer.AdapterPool(2, 16, 64, 48)
    A = np.zeros((8, 64), np.uint16)
    with pytest.raises(mlora.MloraError) as e:           # widths must add up to D
        mlora.mlora_load_adapter_sliced(pool.handle, 0, [A, A], [np.zeros((20, 8), np.uint16)] * 2, 8, 16.0, False)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(mlora.MloraError) as e:           # 3 slices x rank 8 > r_max 16
        mlora.mlora_load_adapter_sliced(pool.handle, 0, [A] * 3, [np.zeros((16, 8), np.uint16)] * 3, 8, 16.0, False)
    assert e.value.status == mlora.MLORA_ERR_RANK_TOO_LARGE
    pool.close()


@pytest.mark.parametrize("T,J,R,seed", [(90, 1, 16, 70), (90, 2, 24, 71), (600, 1, 64, 72), (600, 3, 16, 73)])
def test_separate_gemm_shrink_expand_entry_points(cuda_device, T, J, R, seed):
    """mlora_base_gemm, then mlora_lora_shrink and mlora_lora_expand (the CUDA-core kernels, one
    call each) give the layer's output."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    rng = np.random.default_rng(seed)
    K, D, S = 264, 200, 9
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 2))
    slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("separate", seed, T, J, S, R, slots, scales, {0: synth.normal_bf16(seed, 11, (T, K), 1.0)},
                        [lin])
    dw = DeviceWorkload(wl)
    dw.build_meta()
    dl = dw.linears[0]
    x = dw.x[0]
    y = layer.base_gemm(x, dl.W)
    mlora.mlora_lora_shrink(dl.pool.handle, dw.meta.handle, x)
    mlora.mlora_lora_expand(dl.pool.handle, dw.meta.handle, y)
    torch.cuda.synchronize()
    dw.meta.status()
    assert_close(y.cpu().numpy(), oracle_rows(wl, lin), "separate entry points")
    dw.close()


def _classed_workload(name, seed, T, J, classes, K, D, runs=False):
    """Adapters of a classed pool: slots numbered class by class, each adapter's rank at most its
    class's rank (some at it); tokens draw random slots (or runs of one slot)."""
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    s = 0
    for n, rc in classes:
        for i in range(n):
            r = rc if i % 2 == 0 else int(rng.integers(1, rc + 1))
            lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                            B=synth.normal_bf16(seed, 3000 + s, (D, r), 0.02),
                                            rank=r, alpha=float(2 * r), rslora=bool(s % 3 == 0))
            s += 1
    S = s
    if runs:
        slots = np.repeat(rng.integers(-1, S, size=(T + 95) // 96), 96)[:T].reshape(T, 1).astype(np.int32)
        slots = np.concatenate([slots] + [rng.integers(-1, S, size=(T, 1)).astype(np.int32)] * (J - 1), axis=1)
    else:
        slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload(name, seed, T, J, S, max(r for _, r in classes), slots, scales,
                        {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])
    wl.classes = list(classes)
    return wl


@pytest.mark.parametrize("T,J,classes,K,D,runs,seed", [
    (64, 1, [(5, 8), (4, 16), (3, 64)], 256, 200, False, 80),          # one M-tile: one-CTA GEMM
    (200, 2, [(7, 8), (6, 16), (5, 64)], 320, 392, False, 81),         # two M-tiles: CTA pairs
    (700, 1, [(43, 8), (43, 16), (42, 64)], 256, 520, True, 82),       # the mixed step's classes
    (900, 3, [(9, 8), (3, 24), (4, 100), (2, 256)], 136, 264, False, 83),   # widths 8 / 32 / 128 / 256
])
def test_rank_class_pools(cuda_device, T, J, classes, K, D, runs, seed):
    """Pools whose slots come in rank classes (compact columns: a rank-8 slot is 8 columns wide,
    eight of them share a 64-column block) against the oracle, on the tensor-core side path."""
    wl = _classed_workload("classes", seed, T, J, classes, K, D, runs)
    dw = DeviceWorkload(wl)
    lay = dw.linears[0].pool.layout()
    widths = [w for n, r in classes for w in [{8: 8, 16: 16, 24: 32, 64: 64, 100: 128, 256: 256}[r]] * n]
    assert lay["slot_width"] == widths
    assert all(off % min(w, 64) == 0 for off, w in zip(lay["slot_off"], lay["slot_width"]))
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])
    dw.close()


def test_rank_class_limits_and_mismatch(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    pool = layer.AdapterPool(0, 0, 64, 32, classes=[(2, 8), (2, 16)])
    A, B = np.zeros((16, 64), np.uint16), np.zeros((32, 16), np.uint16)
    with pytest.raises(mlora.MloraError) as e:               # slot 1 is a rank-8 slot
        mlora.mlora_load_adapter(pool.handle, 1, A, B, 16, 32.0, False)
    assert e.value.status == mlora.MLORA_ERR_RANK_TOO_LARGE and "16" in str(e.value) and "8" in str(e.value)
    mlora.mlora_load_adapter(pool.handle, 2, A, B, 16, 32.0, False)     # a rank-16 slot
    other = layer.AdapterPool(4, 16, 64, 32)                 # same slot count, one class
    meta = layer.StepMeta(8, 1, 16)
    meta.build(torch.full((8, 1), -1, dtype=torch.int32, device="cuda"), None, pool)
    x = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mlora.MloraError) as e:
        layer.linear(other, meta, x, W)
    assert e.value.status == mlora.MLORA_ERR_MISMATCH
    for bad in ([(0, 8)], [(2, 0)], [(2, 300)], [(1, 8)] * 9):
        with pytest.raises(mlora.MloraError) as e:
            layer.AdapterPool(0, 0, 64, 32, classes=bad)
        assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    meta.close()
    other.close()
    pool.close()


def test_tiles_past_the_unit_limit_take_the_cuda_core_kernels(cuda_device):
    """J = 8 over 300 rank-64 slots: an M-tile's pairs use more than 256 of the 300 column blocks,
    so the tile overflows the unit lists and its pairs take the CUDA-core shrink and expand; a
    run of one slot keeps other tiles on the tensor cores."""
    rng = np.random.default_rng(90)
    T, J, S, R, K, D = 400, 8, 300, 64, 128, 136
    lin = synth.Linear("lin", K, D, synth.normal_bf16(90, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(90, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(90, 3000 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 2))
    slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    slots[:128] = -1
    slots[:128, 0] = 7                                           # tile 0: one unit
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    wl = synth.Workload("unit-overflow", 90, T, J, S, R, slots, scales,
                        {0: synth.normal_bf16(90, 11, (T, K), 1.0)}, [lin])
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    _check_linear(wl, dw, dw.linears[0])
    dw.close()
