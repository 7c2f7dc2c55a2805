import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the CUDA library")


def read_golden(name: str) -> list:
    """Lines of a golden fixture as (key, [tokens]) pairs, comments and blanks dropped."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *rest = line.split()
                out.append((key, rest))
    return out


@pytest.fixture(scope="session")
def cuda_device():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture
def skinny_form():
    """Sets the small-batch GEMM form for one test (mlora_set_skinny_form), automatic afterwards."""
    from rank_adapter_gemm_token_gb300 import mlora
    yield mlora.mlora_set_skinny_form
    mlora.mlora_set_skinny_form(0)
