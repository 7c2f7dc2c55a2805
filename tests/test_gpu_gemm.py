"""tcgen05 base GEMM against the oracle (no adapters): tile edges, ragged tails, decode and
prefill shapes."""
import numpy as np
import pytest

import oracle
import synth
from tests.harness import assert_close

pytestmark = pytest.mark.gpu


def _run(T, K, D, seed):
    from rank_adapter_gemm_token_gb300 import layer
    x = synth.normal_bf16(seed, 1, (T, K), 1.0)
    W = synth.normal_bf16(seed, 2, (D, K), 0.02)
    y = layer.base_gemm(layer.bf16_from_bits(x, "cuda"), layer.bf16_from_bits(W, "cuda"))
    return x, W, y.cpu().numpy()


@pytest.mark.parametrize("T,K,D", [(1, 8, 16), (16, 256, 256), (127, 64, 64), (129, 72, 200), (300, 200, 520),
                                   (256, 4096, 264), (1000, 512, 1100), (64, 1032, 4096)])
def test_small_and_ragged_shapes(cuda_device, T, K, D):
    x, W, y = _run(T, K, D, seed=T * 7 + D)
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1)
    assert_close(y, ref, f"gemm {T}x{K}x{D}")


@pytest.mark.parametrize("T,K,D", [(256, 4096, 4096), (4096, 4096, 2048), (1024, 14336, 4096)])
def test_large_shapes_sampled(cuda_device, T, K, D):
    x, W, y = _run(T, K, D, seed=D + K)
    rows = np.unique(np.r_[0, T - 1, np.random.default_rng(0).integers(0, T, 30)])
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1, rows=rows)
    assert_close(y[rows], ref, f"gemm {T}x{K}x{D}")


def test_small_integers_are_exact(cuda_device):
    # Small integers in bf16 give exact fp32 products and sums: the GPU must equal the oracle bit for bit.
    from rank_adapter_gemm_token_gb300 import layer
    rng = np.random.default_rng(5)
    T, K, D = 200, 320, 136
    xf = rng.integers(-3, 4, size=(T, K)).astype(np.float32)
    Wf = rng.integers(-3, 4, size=(D, K)).astype(np.float32)
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731  (exact for small ints)
    y = layer.base_gemm(layer.bf16_from_bits(bits(xf), "cuda"), layer.bf16_from_bits(bits(Wf), "cuda")).cpu().numpy()
    ref = oracle.linear(bits(xf), bits(Wf), np.full((T, 1), -1), {}, 1)
    assert np.array_equal(y.astype(np.float64), ref)
