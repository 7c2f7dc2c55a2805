"""The allocation-free entry point (mlora_lora_apply_noalloc) against the pool/metadata path.

Callers that cannot allocate device memory (for example a serving engine that gave all free
device memory to its KV cache at start-up, or a latency-critical path that cannot afford the
device synchronisation of cudaMalloc/cudaFree) use this entry point: it works on their own
buffers plus a fixed workspace compiled into the library. The test runs it twice in a row
through the C ABI and compares each result with mlora_linear on the same inputs."""
import numpy as np
import pytest

import synth
from tests.harness import DeviceWorkload, assert_close

pytestmark = pytest.mark.gpu


def _workload(seed, T=96, K=512, D=384, S=9, R=16, J=2):
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1))
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 2))
    slots = rng.integers(-1, S, size=(T, J)).astype(np.int32)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32)
    return synth.Workload("noalloc", seed, T, J, S, R, slots, scales,
                          {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])


def test_noalloc_matches_the_pool_path_twice(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    for call, seed in enumerate((21, 22)):               # two calls in a row, different inputs
        wl = _workload(seed)
        dw = DeviceWorkload(wl)
        dw.run()
        dw.meta.status()
        dl = dw.linears[0]
        expect = dl.y.clone()
        info = dl.pool.info()
        y = layer.base_gemm(dw.x[0], dl.W)
        mlora.mlora_lora_apply_noalloc(dw.x[0], y, dw.token_slots, dw.scales, wl.T, wl.J, info["A_pool"],
                                       info["B_pool"], info["slot_scale"], info["slot_rank"], info["n_slots"],
                                       info["r_pad"], info["K"], info["D"], torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), expect.cpu().numpy().astype(np.float64), f"no-alloc call {call + 1}")
        dw.close()


def test_noalloc_rejects_sizes_beyond_its_workspace(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import mlora
    T, J, R = 70000, 1, 16                                   # 1,120,000 > 1,048,576 floats
    x = torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_lora_apply_noalloc(x, x, x, None, T, J, x, x, x, x, 4, R, 8, 8)
    assert e.value.status == mlora.MLORA_ERR_TOO_MANY_TOKENS
