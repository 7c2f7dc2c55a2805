"""The adapter cache on the GPU: adapters registered by id in host memory, slots assigned per step
with LRU eviction, missing adapters loaded into every pool of the model; each step's layer
outputs checked against the oracle with the adapters the ids name."""
import numpy as np
import pytest

import oracle
import synth
from tests.harness import assert_close

pytestmark = pytest.mark.gpu

LINEARS = ((256, 128), (128, 256))      # (K, D) of the model's two adapted linears
S, R_MAX, T = 4, 16, 40


def _adapter(seed, i, p, K, D, version=0):
    r = (4, 8, 16)[i % 3]
    return synth.Adapter(A=synth.normal_bf16(seed, 1000 + 100 * version + 10 * i + p, (r, K), 0.02),
                         B=synth.normal_bf16(seed, 5000 + 100 * version + 10 * i + p, (D, r), 0.02),
                         rank=r, alpha=float(2 * r), rslora=bool(i % 2))


def test_adapter_cache_steps(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    seed = 77
    rng = np.random.default_rng(seed)
    pools = [layer.AdapterPool(S, R_MAX, K, D) for K, D in LINEARS]
    Ws = [synth.normal_bf16(seed, 10 + p, (D, K), 0.02) for p, (K, D) in enumerate(LINEARS)]
    xs = [synth.normal_bf16(seed, 20 + p, (T, K), 1.0) for p, (K, D) in enumerate(LINEARS)]
    cache = mlora.mlora_adapter_cache_create([p.handle for p in pools])
    registered = {}
    for i in range(9):
        ads = [_adapter(seed, i, p, K, D) for p, (K, D) in enumerate(LINEARS)]
        registered[100 + i] = ads
        mlora.mlora_adapter_cache_register(cache, 100 + i, [a.A for a in ads], [a.B for a in ads], ads[0].rank,
                                           ads[0].alpha, ads[0].rslora)
    meta = layer.StepMeta(T, 1, R_MAX)

    def step(ids_per_token, expect_loads):
        slots, n_loaded = mlora.mlora_adapter_cache_map(cache, ids_per_token)
        assert n_loaded == expect_loads
        meta.build(torch.from_numpy(slots.reshape(T, 1).copy()).cuda(), None, pools[0])
        for p, (K, D) in enumerate(LINEARS):
            y = layer.linear(pools[p], meta, layer.bf16_from_bits(xs[p], "cuda"), layer.bf16_from_bits(Ws[p], "cuda"))
            by_slot = {int(s): registered[int(i)][p] for i, s in zip(ids_per_token, slots) if i >= 0}
            ref = oracle.linear(xs[p], Ws[p], slots.reshape(T, 1), by_slot, S)
            assert_close(y.cpu().numpy(), ref, f"linear {p}")
        meta.status()
        return slots

    ids = rng.choice([100, 101, 102, -1], size=T)
    step(ids, 3)                                      # three adapters loaded
    step(ids, 0)                                      # all resident
    ids2 = rng.choice([101, 103, 104, -1], size=T)
    s2 = step(ids2, 2)                                # 103 takes the free slot, 104 evicts 100 or 102
    assert len(set(s2[ids2 >= 0].tolist())) == 3
    # a new version of 101: registering again drops the resident copy; the next step loads it
    new = [_adapter(seed, 1, p, K, D, version=1) for p, (K, D) in enumerate(LINEARS)]
    registered[101] = new
    mlora.mlora_adapter_cache_register(cache, 101, [a.A for a in new], [a.B for a in new], new[0].rank,
                                       new[0].alpha, new[0].rslora)
    step(ids2, 1)
    with pytest.raises(mlora.MloraError) as e:        # five distinct adapters, four slots
        mlora.mlora_adapter_cache_map(cache, [100, 101, 102, 103, 104])
    assert e.value.status == mlora.MLORA_ERR_NO_FREE_SLOT
    with pytest.raises(mlora.MloraError) as e:        # not registered
        mlora.mlora_adapter_cache_map(cache, [999])
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    mlora.mlora_adapter_cache_destroy(cache)
    meta.close()
    for p in pools:
        p.close()
