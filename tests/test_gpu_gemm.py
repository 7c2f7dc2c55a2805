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


@pytest.mark.parametrize("T,K,D", [(1900, 328, 2504), (2048, 512, 4864)])
def test_pair_tile_shapes(cuda_device, T, K, D):
    # at least 76 tiles of 256 x 256: the CTA-pair kernel; ragged T (odd 128-row tile count), K, D
    x, W, y = _run(T, K, D, seed=T + K + D)
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1)
    assert_close(y, ref, f"gemm {T}x{K}x{D}")


@pytest.fixture
def gemm_tile():
    from rank_adapter_gemm_token_gb300 import mlora
    yield mlora.mlora_set_gemm_tile_n
    mlora.mlora_set_gemm_tile_n(0)


@pytest.mark.parametrize("bn,D", [(256, 1000), (224, 1000), (192, 1000), (128, 1000), (-1, 1000),
                                  (224, 960), (192, 1024)])
def test_every_gemm_tile_choice(cuda_device, gemm_tile, bn, D):
    # each N tile of the CTA-pair kernel (and the one-CTA kernel, -1) on ragged shapes; D = 960
    # (224) and 1024 (192) end in a tile of two real 32-column store boxes followed by boxes past
    # the edge. Repeated launches must agree bit for bit.
    from rank_adapter_gemm_token_gb300 import layer
    gemm_tile(bn)
    T, K = 1500, 328
    x, W, y = _run(T, K, D, seed=bn + D)
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1)
    assert_close(y, ref, f"gemm {T}x{K}x{D} tile {bn}")
    xd, Wd = layer.bf16_from_bits(x, "cuda"), layer.bf16_from_bits(W, "cuda")
    for _ in range(3):
        assert np.array_equal(layer.base_gemm(xd, Wd).cpu().numpy(), y), "GEMM result differs between launches"


@pytest.mark.parametrize("T,K,D", [(256, 4096, 4096), (4096, 4096, 2048), (1024, 14336, 4096)])
def test_large_shapes_sampled(cuda_device, T, K, D):
    x, W, y = _run(T, K, D, seed=D + K)
    rows = np.unique(np.r_[0, T - 1, np.random.default_rng(0).integers(0, T, 30)])
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1, rows=rows)
    assert_close(y[rows], ref, f"gemm {T}x{K}x{D}")


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("T,K,D", [(1, 64, 520), (17, 328, 4100), (250, 200, 2056), (64, 1032, 4096),
                                   (256, 4096, 4096)])
def test_small_batch_gemm_forms(cuda_device, skinny_form, form, T, K, D):
    # both forms of the small-batch GEMM (split-K CTA pairs; token groups sharing W and x rows by
    # multicast) on ragged token counts and a partial last output block; deterministic
    from rank_adapter_gemm_token_gb300 import layer
    skinny_form(form)
    x, W, y = _run(T, K, D, seed=T + D + form)
    rows = None if T * D <= 600_000 else np.unique(np.r_[0, T - 1, np.random.default_rng(1).integers(0, T, 30)])
    ref = oracle.linear(x, W, np.full((T, 1), -1), {}, 1, rows=rows)
    assert_close(y if rows is None else y[rows], ref, f"gemm {T}x{K}x{D} form {form}")
    xd, Wd = layer.bf16_from_bits(x, "cuda"), layer.bf16_from_bits(W, "cuda")
    assert np.array_equal(layer.base_gemm(xd, Wd).cpu().numpy(), y), "GEMM result differs between launches"


@pytest.mark.parametrize("T,K,D", [(200, 320, 136), (1900, 200, 2600)])
def test_small_integers_are_exact(cuda_device, T, K, D):
    # Small integers in bf16 give exact fp32 products and sums: the GPU must equal the oracle bit
    # for bit (small-batch CTA-pair kernel; large-batch CTA-pair kernel with a ragged last pair tile).
    from rank_adapter_gemm_token_gb300 import layer
    rng = np.random.default_rng(5)
    xf = rng.integers(-3, 4, size=(T, K)).astype(np.float32)
    Wf = rng.integers(-3, 4, size=(D, K)).astype(np.float32)
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731  (exact for small ints)
    y = layer.base_gemm(layer.bf16_from_bits(bits(xf), "cuda"), layer.bf16_from_bits(bits(Wf), "cuda")).cpu().numpy()
    ref = oracle.linear(bits(xf), bits(Wf), np.full((T, 1), -1), {}, 1)
    assert np.array_equal(y.astype(np.float64), ref)
