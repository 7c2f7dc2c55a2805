"""Edge cases of the layer on the GPU against the fp64 oracle: an empty batch, the largest rank
and slots-per-token limits, a 2048-slot pool, and the batch sizes on both sides of the switch
from the small-batch path (fused shrink, T <= 256) to the large-batch paths."""
import numpy as np
import pytest

import synth
from tests.harness import DeviceWorkload, assert_close, oracle_rows

pytestmark = pytest.mark.gpu


def _workload(name, seed, T, K, D, S, R, J, ranks, sentinel_every=4, load=None):
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in (range(S) if load is None else load):
        r = int(ranks(s, rng))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 5000 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 2 == 0))
    loaded = np.array(sorted(lin.adapters), dtype=np.int32)
    slots = loaded[rng.integers(0, len(loaded), size=(T, J))].astype(np.int32)
    slots[rng.uniform(size=(T, J)) < 0.25] = -1
    slots[::sentinel_every, :] = -1
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    return synth.Workload(name, seed, T, J, S, R, slots, scales, {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])


def _run_and_check(wl):
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    dl = dw.linears[0]
    assert_close(dl.y.cpu().numpy(), oracle_rows(wl, dl.lin), wl.name)
    dw.close()


def test_empty_batch_writes_nothing(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    pool = layer.AdapterPool(4, 8, 64, 32)
    meta = layer.StepMeta(16, 1, 8)
    meta.build(torch.zeros((0, 1), dtype=torch.int32, device="cuda"), None, pool)
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.full((1, 32), 7.0, device="cuda")              # a buffer the call must not touch
    mlora.mlora_linear(pool.handle, meta.handle, x, W, y[:0], None)
    torch.cuda.synchronize()
    meta.status()
    assert torch.all(y == 7.0)
    pool.close()
    meta.close()


def test_eight_slots_per_token_and_the_largest_rank(cuda_device):
    # J = 8 (the limit), r_max = 256 (the limit): one adapter at rank 256, others spread below
    wl = _workload("j8-r256", 21, T=90, K=136, D=72, S=12, R=256, J=8,
                   ranks=lambda s, rng: 256 if s == 3 else rng.integers(1, 200))
    _run_and_check(wl)


@pytest.mark.parametrize("T", [256, 257])
def test_small_batch_switch(cuda_device, T):
    # 256 tokens take the fused small-batch path, 257 the tensor-core side path (three M-tiles of
    # per-token random slots)
    wl = _workload(f"switch-{T}", 30 + T, T=T, K=520, D=264, S=20, R=64, J=1,
                   ranks=lambda s, rng: (8, 16, 64)[s % 3])
    _run_and_check(wl)


def test_pool_of_2048_slots(cuda_device):
    # the slot limit; 300 of the 2048 slots hold adapters, spread over the whole id range
    load = sorted(np.random.default_rng(7).choice(2048, size=300, replace=False).tolist())
    wl = _workload("s2048", 40, T=600, K=64, D=48, S=2048, R=16, J=2,
                   ranks=lambda s, rng: rng.integers(1, 17), load=load)
    _run_and_check(wl)
