"""The C-ABI library builds for sm_103a, loads, and exports every entry point mlora.h declares.
No compute call is made here (this runs without a GPU)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT, read_golden


@pytest.fixture(scope="module")
def lib():
    from rank_adapter_gemm_token_gb300 import build, mlora
    build.build()
    return mlora.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "mlora.h")).read()
    return sorted(set(re.findall(r"MLORA_API [^;(]*?\b(mlora_\w+)\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("mlora_pool_create", "mlora_load_adapter", "mlora_build_meta", "mlora_linear",
                     "mlora_pool_bytes", "mlora_meta_status", "mlora_status_string", "mlora_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from rank_adapter_gemm_token_gb300 import mlora
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in mlora.h but not exported"
    assert set(_declared()) == set(mlora.EXPORTS)


def test_only_the_abi_is_exported(lib):
    import subprocess
    from rank_adapter_gemm_token_gb300 import mlora
    out = subprocess.run(["nm", "-D", "--defined-only", mlora.library_path()], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert {n for n in exported if n.startswith("mlora_")} == set(_declared())


def test_pool_bytes_reproduces_the_pages_slot_figures(lib):
    # "Multi-LoRA Serving Explained": slot memory = slots * adapter size at the maximum rank,
    # adapters spanning 32 blocks x 7 linears of the made-up model.
    from oracle import memory
    from rank_adapter_gemm_token_gb300 import mlora
    GiB, MiB = 2.0 ** 30, 2.0 ** 20

    def model_slots(n, r):
        return memory.LAYERS * sum(mlora.mlora_pool_bytes(n, r, i, o) for i, o in memory.MODULES.values())

    for key, v in read_golden("memory_figures.txt"):
        if key == "slots_gib":
            assert round(model_slots(int(v[0]), int(v[1])) / GiB, int(v[3])) == float(v[2])
        elif key == "adapter_mib":
            assert round(model_slots(1, int(v[0])) / MiB, int(v[2])) == float(v[1])
        elif key == "hundred_rank16_gib":
            assert round(model_slots(100, 16) / GiB, int(v[1])) == float(v[0])
    assert mlora.mlora_pool_bytes(0, 8, 64, 64) == 0
    assert mlora.mlora_pool_bytes(1, 5, 64, 64) == 1 * 8 * 128 * 2      # slot width 8
    assert mlora.mlora_pool_bytes(2, 24, 64, 64) == 2 * 32 * 128 * 2     # 8, 16, 32, 64 ...
    assert mlora.mlora_pool_bytes(1, 100, 64, 64) == 1 * 128 * 128 * 2   # ... then multiples of 64


def test_status_strings(lib):
    from rank_adapter_gemm_token_gb300 import mlora
    assert mlora.mlora_status_string(0) == "ok"
    assert "rank" in mlora.mlora_status_string(mlora.MLORA_ERR_RANK_TOO_LARGE)
    assert mlora.mlora_kernel_kind_name(1) == "base_gemm"
    assert mlora.mlora_version() >= 1


def test_null_arguments_are_rejected_without_a_device(lib):
    from rank_adapter_gemm_token_gb300 import mlora
    assert lib.mlora_pool_create(4, 8, 64, 64, None, None) == mlora.MLORA_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    assert lib.mlora_pool_create(0, 8, 64, 64, None, ctypes.byref(out)) == mlora.MLORA_ERR_INVALID_ARG
    assert lib.mlora_pool_create(4, 8, 60, 64, None, ctypes.byref(out)) == mlora.MLORA_ERR_INVALID_ARG
    assert lib.mlora_meta_create(0, 1, 8, ctypes.byref(out)) == mlora.MLORA_ERR_INVALID_ARG
    assert lib.mlora_load_adapter(None, 0, None, None, 4, 8.0, 0) == mlora.MLORA_ERR_INVALID_ARG
    assert lib.mlora_linear(None, None, None, None, None, None) == mlora.MLORA_ERR_INVALID_ARG


def test_no_gpu_means_a_loud_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from rank_adapter_gemm_token_gb300 import mlora
    with pytest.raises(mlora.MloraError) as e:
        mlora.mlora_pool_create(4, 8, 64, 64)
    assert e.value.status == mlora.MLORA_ERR_CUDA


def test_missing_library_fails_loudly(tmp_path):
    from rank_adapter_gemm_token_gb300 import mlora
    with pytest.raises(FileNotFoundError):
        mlora.load(str(tmp_path / "libmlora.so"))


def test_gemm_tile_choice_is_validated(lib):
    from rank_adapter_gemm_token_gb300 import mlora
    for n in (256, 224, 192, 128, -1, 0):
        assert lib.mlora_set_gemm_tile_n(n) == mlora.MLORA_OK
    for n in (1, 64, 160, 512, -2):
        assert lib.mlora_set_gemm_tile_n(n) == mlora.MLORA_ERR_INVALID_ARG
    assert lib.mlora_set_gemm_tile_n(0) == mlora.MLORA_OK


def test_path_and_small_batch_form_choices_are_validated(lib):
    from rank_adapter_gemm_token_gb300 import mlora
    for setter, good, bad in ((lib.mlora_set_path, (0, 1, 2), (-1, 3)),
                              (lib.mlora_set_skinny_form, (0, 1, 2), (-1, 3, 7))):
        for v in good:
            assert setter(v) == mlora.MLORA_OK
        for v in bad:
            assert setter(v) == mlora.MLORA_ERR_INVALID_ARG
        assert setter(0) == mlora.MLORA_OK
