"""Failure path without a GPU fault.

A kernel whose wait runs out returns on its own, the host reads FA_ERR_TIMEOUT,
and the context stays usable.  Two forms:
- a probe kernel that waits on a barrier nothing completes;
- the real forward and backward kernels, made to abort through
  fa_debug_abort_next_call(): the MMA-issuing role acts as if its first wait had
  timed out and raises the abort flag; every other role leaves its loop through its
  own bounded wait, drains the copies and products it issued, frees tensor memory
  and returns.  A normal call after it must still match the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import attention_dense, attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, f64, max_abs, o_within_bar, rel_fro, require_gpu

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_wait_timeout_is_reported_and_context_survives():
    from exact_attention_flash_gb300 import _lib, fa_get_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    lib = _lib.load()
    assert fa_get_device_status() == 0
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fa_debug_wait_timeout(2_000_000, stream) == 0  # 2 ms limit; nothing ever arrives
    assert fa_get_device_status() == FA_ERR_TIMEOUT  # read and cleared
    assert fa_get_device_status() == 0
    q, k, v, _ = make_attention_inputs(1, 1, 256, 64, 0, "cuda", with_do=False)
    o, lse = fa_forward(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert fa_get_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_forward_abort_path_then_normal_call(d):
    """The persistent forward (B = H = 1, N = 256), made to abort, comes back with
    FA_ERR_TIMEOUT; the next call on the same buffers and workspace is exact."""
    from exact_attention_flash_gb300 import _lib, fa_forward, fa_get_device_status, forward_workspace_bytes
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    lib = _lib.load()
    assert fa_get_device_status() == 0
    q, k, v, _ = make_attention_inputs(1, 1, 256, d, 300 + d, "cuda", with_do=False)
    ws = torch.empty(forward_workspace_bytes(1, 1, 256, d, True), device="cuda", dtype=torch.uint8)
    o = torch.empty((1, 1, 256, d), device="cuda", dtype=torch.float32)
    lse = torch.empty((1, 1, 256), device="cuda")
    assert lib.fa_debug_abort_next_call() == 0
    fa_forward(q, k, v, causal=True, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert fa_get_device_status() == FA_ERR_TIMEOUT
    assert fa_get_device_status() == 0
    fa_forward(q, k, v, causal=True, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert fa_get_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v), causal=True)
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS


@pytest.mark.parametrize("d", [64, 128])
def test_backward_abort_path_then_normal_call(d):
    """The backward (preprocess + main kernel, B = H = 1, N = 256), made to abort,
    comes back with FA_ERR_TIMEOUT; the next call is exact."""
    from exact_attention_flash_gb300 import _lib, fa_backward, fa_forward, fa_get_device_status
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    lib = _lib.load()
    q, k, v, do = make_attention_inputs(1, 1, 256, d, 310 + d, "cuda")
    o, lse = fa_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa_get_device_status() == 0
    assert lib.fa_debug_abort_next_call() == 0
    fa_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa_get_device_status() == FA_ERR_TIMEOUT
    assert fa_get_device_status() == 0
    dq, dk, dv = fa_backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa_get_device_status() == 0
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        g = f64(g)
        assert np.isfinite(g).all(), name
        assert rel_fro(g, r) <= GRAD_REL_FRO, name


def test_abort_flag_applies_to_one_call_only():
    """The flag is taken by the next call: the calls after it run normally."""
    from exact_attention_flash_gb300 import _lib, fa_forward, fa_get_device_status
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    lib = _lib.load()
    q, k, v, _ = make_attention_inputs(2, 2, 300, 128, 320, "cuda", with_do=False)
    assert lib.fa_debug_abort_next_call() == 0
    fa_forward(q, k, v)
    torch.cuda.synchronize()
    assert fa_get_device_status() == FA_ERR_TIMEOUT
    for _ in range(3):
        o, lse = fa_forward(q, k, v)
        torch.cuda.synchronize()
        assert fa_get_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v))
    assert o_within_bar(f64(o), ref_o, "bf16") <= 0.0
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS
