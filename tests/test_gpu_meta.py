"""GPU slot metadata against the oracle's stable sort: bit-exact order, segments and counts."""
import numpy as np
import pytest

import oracle
from tests.conftest import read_golden

pytestmark = pytest.mark.gpu


def _pool(n_slots, K=64, D=64, r_max=8, loaded=None):
    from rank_adapter_gemm_token_gb300 import layer
    pool = layer.AdapterPool(n_slots, r_max, K, D)
    A = np.zeros((1, K), dtype=np.uint16)
    B = np.zeros((D, 1), dtype=np.uint16)
    for s in (range(n_slots) if loaded is None else loaded):
        pool.load(s, A, B, 1, 1.0)
    pool.sync()
    return pool


def _meta_on_gpu(ids, n_slots, pool=None, scales=None):
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    ids = np.asarray(ids, dtype=np.int32)
    if ids.ndim == 1:
        ids = ids.reshape(-1, 1)
    T, J = ids.shape
    pool = pool or _pool(n_slots)
    meta = layer.StepMeta(max(T, 1), J, 8)
    dev = torch.from_numpy(np.ascontiguousarray(ids)).cuda()
    meta.build(dev, scales, pool)
    return meta, pool


def test_six_token_example(cuda_device):
    g = dict(read_golden("segments_six_tokens.txt"))
    ids = [int(v) for v in g["ids"]]
    meta, pool = _meta_on_gpu(ids, 4)
    meta.status()
    got = meta.read()
    assert got == oracle.meta(np.array(ids).reshape(-1, 1), 4)
    assert got["order"] == [int(v) for v in g["order"]]


@pytest.mark.parametrize("T,J,S,seed", [(1, 1, 1, 0), (37, 1, 5, 1), (256, 1, 100, 2), (128, 3, 32, 3),
                                        (1023, 2, 7, 4), (1024, 1, 128, 5), (1500, 3, 2048, 6), (4096, 1, 8, 7)])
def test_random_ids_match_the_stable_sort(cuda_device, T, J, S, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    meta, pool = _meta_on_gpu(ids, S)
    meta.status()
    assert meta.read() == oracle.meta(ids, S)


def test_all_sentinel_and_empty_steps(cuda_device):
    meta, pool = _meta_on_gpu(np.full((40, 2), -1), 3)
    meta.status()
    m = meta.read()
    assert m == oracle.meta(np.full((40, 2), -1), 3) and m["n_active"] == 0
    meta2, _ = _meta_on_gpu(np.zeros((0, 1), dtype=np.int32), 3, pool=pool)
    meta2.status()
    assert meta2.read()["n_active"] == 0


def test_bad_and_empty_slot_ids_are_reported(cuda_device):
    from rank_adapter_gemm_token_gb300 import mlora
    pool = _pool(6, loaded=[0, 1, 2, 4, 5])            # slot 3 never loaded
    for bad in (6, -2, 3):
        ids = np.array([[0], [1], [bad], [2]], dtype=np.int32)
        meta, _ = _meta_on_gpu(ids, 6, pool=pool)
        with pytest.raises(mlora.MloraError) as e:
            meta.status()
        assert e.value.status == mlora.MLORA_ERR_BAD_TOKEN_SLOT
        assert "pair 2" in str(e.value)
        # the rejected pair is treated as the sentinel, nothing else changes
        fixed = ids.copy()
        fixed[2, 0] = -1
        assert meta.read() == oracle.meta(fixed, 6)
        meta.status()                                  # the error word was cleared


def test_too_many_tokens(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    pool = _pool(2)
    meta = layer.StepMeta(8, 1, 8)
    with pytest.raises(mlora.MloraError) as e:
        meta.build(torch.zeros((9, 1), dtype=torch.int32, device="cuda"), None, pool)
    assert e.value.status == mlora.MLORA_ERR_TOO_MANY_TOKENS
