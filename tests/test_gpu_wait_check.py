"""Failure detection without a GPU fault: a kernel whose bounded wait can never complete gives up
after the library's limit, reports MLORA_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import time

import pytest

import synth
from tests.harness import DeviceWorkload, assert_close, oracle_rows

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_stays_usable(cuda_device):
    import torch
    from rank_adapter_gemm_token_gb300 import mlora
    t0 = time.monotonic()
    status = mlora.mlora_check_wait_timeout()
    elapsed = time.monotonic() - t0
    assert status == mlora.MLORA_ERR_DEVICE_TIMEOUT, mlora.mlora_last_error()
    assert 1.5 < elapsed < 30.0, f"the wait should give up after about 2 s, took {elapsed:.1f} s"
    # the library-wide error word is untouched and the GPU still computes correctly
    wl = synth.tiny()
    dw = DeviceWorkload(wl)
    dw.run()
    dw.meta.status()
    dl = dw.linears[0]
    assert_close(dl.y.cpu().numpy(), oracle_rows(wl, dl.lin), "after the wait check")
    dw.close()
    torch.cuda.synchronize()
