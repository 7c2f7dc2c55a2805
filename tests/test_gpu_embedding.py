"""The embedding lookup with LoRA (mlora_embedding) against the fp64 oracle, element by element.

Tolerance, from the arithmetic: a table entry is a bf16 value, exact in fp32; the side path adds
at most 256 products of bf16 values (each exact in fp32) times a scaled fp32 factor, summed in
fp32, so its error is below (r + 2) 2^-24 times the sum of the terms' magnitudes, about 3e-6 for
the largest cases here. The tests allow 2e-5 absolute and 1e-5 relative Frobenius, and demand
exact equality with the table row where every slot of a token is -1."""
import numpy as np
import pytest

import oracle
import synth
from tests.harness import assert_close

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5
ABS_TOL = 2e-5


class _Device:
    """An embedding workload on the GPU: pool, table, ids, token slots, scales, metadata."""

    def __init__(self, wl, J_meta=None):
        import torch
        from rank_adapter_gemm_token_gb300 import layer
        self.torch, self.layer, self.wl = torch, layer, wl
        self.pool = layer.EmbeddingPool(wl.vocab, wl.dim, wl.classes)
        for s, ad in wl.adapters.items():
            self.pool.load(s, ad.A, ad.B, ad.rank, ad.alpha, ad.rslora)
        self.pool.sync()
        self.E = layer.bf16_from_bits(wl.E, "cuda")
        self.ids = torch.from_numpy(np.ascontiguousarray(wl.ids.astype(np.int32))).cuda()
        self.slots = torch.from_numpy(np.ascontiguousarray(wl.token_slots.astype(np.int32))).cuda()
        self.scales = None if wl.scales is None else torch.from_numpy(np.ascontiguousarray(wl.scales)).cuda()
        self.meta = layer.StepMeta(max(wl.T, 1), J_meta or wl.J, wl.r_max)

    def run(self):
        self.meta.build(self.slots, self.scales, self.pool)
        y = self.layer.embedding(self.pool, self.meta, self.ids, self.E)
        self.torch.cuda.synchronize()
        return y

    def close(self):
        self.pool.close()
        self.meta.close()


def _reference(wl, rows=None):
    return oracle.embedding(wl.ids, wl.E, wl.token_slots, wl.adapters, wl.n_slots, scales=wl.scales, rows=rows)


def _check(wl, y, what):
    y = y.cpu().numpy()
    ref = _reference(wl)
    assert_close(y, ref, what, rel_tol=REL_TOL, abs_tol=ABS_TOL)
    none = np.all(wl.token_slots < 0, axis=1)
    table = synth.bf16_bits_to_f32(wl.E[wl.ids[none]])
    assert np.array_equal(y[none], table), f"{what}: rows without an adapter differ from the table"


@pytest.mark.parametrize("T,vocab,dim,J,classes,scales", [
    (300, 1000, 264, 1, [(6, 8), (5, 16), (3, 64)], True),      # ragged column range, three classes
    (77, 517, 130, 3, [(8, 16)], True),                           # several slots per token
    (513, 4099, 1030, 2, [(4, 32), (2, 256)], False),             # rank 256, no scales
    (1, 50, 2, 1, [(1, 8)], True),                                # one token, two columns
    (2048, 3001, 520, 1, [(40, 16)], True),                       # many pair-blocks and sentinel groups
    (96, 700, 4096, 8, [(3, 8), (9, 64)], True),                  # eight slots per token, full width
    (200, 777, 264, 1, [(3, 128), (2, 8)], True),                 # one slot per token, slots wider than 64
])
def test_embedding_matches_the_oracle(cuda_device, T, vocab, dim, J, classes, scales):
    wl = synth.embedding_case(T, vocab, dim, J, classes, with_scales=scales)
    dev = _Device(wl)
    y = dev.run()
    dev.meta.status()
    _check(wl, y, f"embedding T={T} V={vocab} D={dim} J={J}")
    dev.close()


def test_embedding_full_size_mixed_step(cuda_device):
    """The mixed serving step's 1024 tokens through a 100000 x 4096 table, 128 slots in three rank
    classes: every row and column against the oracle."""
    wl = synth.embedding_step()
    dev = _Device(wl)
    y = dev.run()
    dev.meta.status()
    _check(wl, y, "embedding, mixed step")
    dev.close()


def test_embedding_slot_reload_and_empty_step(cuda_device):
    """A slot cleared and reloaded with a smaller adapter (the scatter must zero the columns past
    the new rank), and a step without tokens."""
    wl = synth.embedding_case(200, 900, 136, 1, [(4, 64)], sentinel_frac=0.0)
    dev = _Device(wl)
    dev.run()
    small = synth.embedding_case(1, 900, 136, 1, [(4, 16)], seed_offset=31).adapters[1]
    dev.pool.clear(2)
    dev.pool.load(2, small.A, small.B, small.rank, small.alpha, small.rslora)
    dev.pool.sync()
    wl.adapters[2] = small
    _check(wl, dev.run(), "embedding after a reload")
    import torch
    empty = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    dev.meta.build(empty, None, dev.pool)
    y = dev.layer.embedding(dev.pool, dev.meta, dev.ids[:0].contiguous(), dev.E)
    torch.cuda.synchronize()
    assert y.shape == (0, wl.dim)
    dev.close()


def test_embedding_reports_ids_outside_the_table(cuda_device):
    from rank_adapter_gemm_token_gb300 import mlora
    wl = synth.embedding_case(64, 300, 72, 2, [(5, 16)])
    dev = _Device(wl)
    dev.ids[5] = wl.vocab                      # one past the table
    dev.ids[9] = -3
    y = dev.run()
    with pytest.raises(mlora.MloraError) as e:
        dev.meta.status()
    assert e.value.status == mlora.MLORA_ERR_BAD_TOKEN_ID
    yh = y.cpu().numpy()
    assert not yh[[5, 9]].any(), "rows of rejected ids must be zero"
    rows = np.array([t for t in range(wl.T) if t not in (5, 9)])
    assert_close(yh[rows], _reference(wl, rows), "embedding rows beside rejected ids", rel_tol=REL_TOL,
                 abs_tol=ABS_TOL)
    dev.meta.status()                          # the error word was cleared
    dev.close()


def test_embedding_pool_is_kept_apart_from_the_linear_calls(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import layer, mlora
    wl = synth.embedding_case(32, 400, 64, 1, [(4, 16)])
    dev = _Device(wl)
    dev.run()
    x = torch.zeros((32, 400), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 400), dtype=torch.bfloat16, device="cuda")
    for call in (lambda: layer.linear(dev.pool, dev.meta, x[:, :400], W),
                 lambda: mlora.mlora_lora_expand(dev.pool.handle, dev.meta.handle, torch.zeros((32, 64), device="cuda"))):
        with pytest.raises(mlora.MloraError) as e:
            call()
        assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    ad = wl.adapters[0]
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_load_adapter_sliced(dev.pool.handle, 0, [ad.A, ad.A], [ad.B[:32], ad.B[32:]], ad.rank, ad.alpha,
                                        False)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    lin_pool = layer.AdapterPool(4, 16, 400, 64)
    lin_pool.load(0, ad.A, ad.B, ad.rank, ad.alpha)
    lin_pool.sync()
    with pytest.raises(mlora.MloraError) as e:
        layer.embedding(lin_pool, dev.meta, dev.ids, dev.E)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_embedding_pool_create([4], [16], 400, 63)
    assert e.value.status == mlora.MLORA_ERR_INVALID_ARG
    lin_pool.close()
    dev.close()


def test_one_meta_serves_the_embedding_and_the_linears(cuda_device):
    """Metadata built once with a linear pool of the same classes drives the embedding too."""
    import torch
    from rank_adapter_gemm_token_gb300 import layer
    wl = synth.embedding_case(150, 640, 256, 1, [(3, 8), (4, 64)])
    dev = _Device(wl)
    lin_pool = layer.AdapterPool(0, 0, 256, 128, classes=wl.classes)
    for s in range(wl.n_slots):
        r = wl.adapters[s].rank
        lin_pool.load(s, synth.normal_bf16(1, 900 + s, (r, 256), 0.02), synth.normal_bf16(1, 950 + s, (128, r), 0.02),
                      r, 2.0 * r)
    lin_pool.sync()
    dev.meta.build(dev.slots, dev.scales, lin_pool)
    y = layer.embedding(dev.pool, dev.meta, dev.ids, dev.E)
    torch.cuda.synchronize()
    dev.meta.status()
    _check(wl, y, "embedding with metadata built on a linear pool")
    lin_pool.close()
    dev.close()
