"""Failure path without a GPU fault: a kernel whose wait runs out returns on its
own, the host reads FA_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    require_gpu()
    from exact_attention_flash_gb300 import _lib, fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    lib = _lib.load()
    assert fa_device_status() == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fa_debug_wait_timeout(2_000_000, stream) == 0  # 2 ms limit; nothing ever arrives
    assert fa_device_status() == 4  # FA_ERR_TIMEOUT, read and cleared
    assert fa_device_status() == 0
    q, k, v, _ = make_attention_inputs(1, 1, 256, 64, 0, "cuda", with_do=False)
    o, lse = fa_forward(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert fa_device_status() == 0
