"""The allocation-free entry point (mlora_lora_apply_noalloc) against the fp64 oracle and the
pool/metadata path.

Some callers of this library cannot allocate device memory when they run the layer: a serving
engine that gave all free device memory to its KV cache at start-up (a later cudaMalloc fails),
or a latency-critical path that cannot afford the device synchronisation of cudaMalloc/cudaFree.
They use this entry point: it works on their own buffers (adapters laid out slot by slot) plus a
fixed workspace compiled into the library. The tests call it through the C ABI: twice in a row
against mlora_linear and the oracle, over rank widths, slots per token, an all-sentinel batch,
a request of exactly the workspace's size, an over-sized rank and no scales, and check that a
call changes no device allocation."""
import numpy as np
import pytest

import oracle
import synth
from tests.harness import DeviceWorkload, assert_close

pytestmark = pytest.mark.gpu


def _workload(seed, T=96, K=512, D=384, S=9, R=16, J=2, sentinel_only=False, with_scales=True):
    rng = np.random.default_rng(seed)
    lin = synth.Linear("lin", K, D, synth.normal_bf16(seed, 10, (D, K), 0.02), 0)
    for s in range(S):
        r = int(rng.integers(1, R + 1)) if s else R               # slot 0 fills the rank width
        lin.adapters[s] = synth.Adapter(A=synth.normal_bf16(seed, 100 + s, (r, K), 0.02),
                                        B=synth.normal_bf16(seed, 300 + s, (D, r), 0.02),
                                        rank=r, alpha=float(2 * r), rslora=bool(s % 2))
    slots = np.full((T, J), -1, np.int32) if sentinel_only else rng.integers(-1, S, size=(T, J)).astype(np.int32)
    scales = rng.uniform(0.2, 1.0, size=(T, J)).astype(np.float32) if with_scales else None
    return synth.Workload("noalloc", seed, T, J, S, R, slots, scales,
                          {0: synth.normal_bf16(seed, 11, (T, K), 1.0)}, [lin])


def _slot_factor(ad) -> np.float32:
    r = np.float32(ad.rank)
    return np.float32(ad.alpha) / (np.sqrt(r) if ad.rslora else r)


def _noalloc_buffers(wl, r_pad):
    """The adapters of the workload's linear laid out slot by slot: A [S, r_pad, K], B [S, D, r_pad]
    (zero beyond each rank), slot factors and ranks, on the GPU."""
    import torch
    lin = wl.linears[0]
    S, K, D = wl.n_slots, lin.K, lin.D
    A = np.zeros((S, r_pad, K), np.uint16)
    B = np.zeros((S, D, r_pad), np.uint16)
    c = np.zeros(S, np.float32)
    rk = np.zeros(S, np.int32)
    for s, ad in lin.adapters.items():
        A[s, :ad.rank] = ad.A
        B[s, :, :ad.rank] = ad.B
        c[s] = _slot_factor(ad)
        rk[s] = ad.rank
    dev = torch.device("cuda")
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    return to(A.view(np.int16)).view(torch.bfloat16), to(B.view(np.int16)).view(torch.bfloat16), to(c), to(rk)


def _apply(wl, r_pad, slot_rank_override=None):
    """y = base product (library GEMM) + the no-alloc side path; returns y on the host."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    lin = wl.linears[0]
    x = layer.bf16_from_bits(wl.xs[0], "cuda")
    W = layer.bf16_from_bits(lin.W, "cuda")
    slots = torch.from_numpy(np.ascontiguousarray(wl.token_slots)).cuda()
    scales = None if wl.scales is None else torch.from_numpy(np.ascontiguousarray(wl.scales)).cuda()
    A, B, c, rk = _noalloc_buffers(wl, r_pad)
    if slot_rank_override is not None:
        rk = torch.from_numpy(slot_rank_override).cuda()
    y = layer.base_gemm(x, W)
    mlora.mlora_lora_apply_noalloc(x, y, slots, scales, wl.T, wl.J, A, B, c, rk, wl.n_slots, r_pad, lin.K, lin.D,
                                   torch.cuda.current_stream())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _reference(wl):
    lin = wl.linears[0]
    return oracle.linear(wl.xs[0], lin.W, wl.token_slots, lin.adapters, wl.n_slots, scales=wl.scales)


def test_noalloc_matches_the_pool_path_and_the_oracle_twice(cuda_device):
    for call, seed in enumerate((21, 22)):               # two calls in a row, different inputs
        wl = _workload(seed)
        dw = DeviceWorkload(wl)
        dw.run()
        dw.meta.status()
        expect = dw.linears[0].y.cpu().numpy().astype(np.float64)
        dw.close()
        y = _apply(wl, 16)
        assert_close(y, expect, f"no-alloc call {call + 1} against mlora_linear")
        assert_close(y, _reference(wl), f"no-alloc call {call + 1} against the oracle")


@pytest.mark.parametrize("r_pad,J", [(16, 1), (64, 3), (256, 8), (8, 2)])
def test_noalloc_rank_widths_and_slots_per_token(cuda_device, r_pad, J):
    wl = _workload(30 + r_pad + J, T=80, K=256, D=200, S=6, R=r_pad, J=J)
    assert_close(_apply(wl, r_pad), _reference(wl), f"no-alloc r_pad={r_pad} J={J}")


def test_noalloc_without_scales_and_all_sentinel(cuda_device):
    wl = _workload(41, T=64, K=128, D=136, S=5, R=16, J=2, with_scales=False)
    assert_close(_apply(wl, 16), _reference(wl), "no-alloc, scales NULL")
    wl = _workload(42, T=64, K=128, D=136, S=5, R=16, J=2, sentinel_only=True)
    y = _apply(wl, 16)
    assert_close(y, _reference(wl), "no-alloc, every slot -1")


def test_noalloc_at_exactly_the_workspace_size(cuda_device):
    T, J, r_pad = 4096, 1, 256                          # T * J * r_pad = 2^20 floats exactly
    assert T * J * r_pad == 1 << 20
    wl = _workload(43, T=T, K=64, D=72, S=4, R=r_pad, J=J)
    assert_close(_apply(wl, r_pad), _reference(wl), "no-alloc at 2^20 workspace floats")


def test_noalloc_ignores_a_rank_above_the_width(cuda_device):
    wl = _workload(44, T=96, K=128, D=96, S=5, R=16, J=1)
    rk = np.array([wl.linears[0].adapters[s].rank for s in range(wl.n_slots)], np.int32)
    rk[2] = 24                                           # more rows than the slot holds: adds nothing
    y = _apply(wl, 16, slot_rank_override=rk)
    cut = synth.Workload(wl.name, wl.seed, wl.T, wl.J, wl.n_slots, wl.r_max,
                         np.where(wl.token_slots == 2, -1, wl.token_slots).astype(np.int32), wl.scales, wl.xs,
                         wl.linears)
    assert_close(y, _reference(cut), "no-alloc with an over-sized rank on slot 2")


def test_noalloc_allocates_nothing(cuda_device):
    import torch
    wl = _workload(45, T=64, K=128, D=128, S=4, R=16, J=2)
    _apply(wl, 16)                                       # the library's module (and workspace) is loaded now
    from rank_adapter_gemm_token_gb300 import layer, mlora
    lin = wl.linears[0]
    x = layer.bf16_from_bits(wl.xs[0], "cuda")
    y = layer.base_gemm(x, layer.bf16_from_bits(lin.W, "cuda"))
    slots = torch.from_numpy(wl.token_slots).cuda()
    scales = torch.from_numpy(wl.scales).cuda()
    A, B, c, rk = _noalloc_buffers(wl, 16)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        mlora.mlora_lora_apply_noalloc(x, y, slots, scales, wl.T, wl.J, A, B, c, rk, wl.n_slots, 16, lin.K, lin.D,
                                       torch.cuda.current_stream())
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_rejects_sizes_beyond_its_workspace(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import mlora
    T, J, R = 70000, 1, 16                                   # 1,120,000 > 1,048,576 floats
    x = torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_lora_apply_noalloc(x, x, x, None, T, J, x, x, x, x, 4, R, 8, 8)
    assert e.value.status == mlora.MLORA_ERR_TOO_MANY_TOKENS
