"""Parity of the general query offset (fa_forward_qk / fa_backward_qk: Nq queries at
positions q_start .. q_start + Nq - 1 against Nk keys) with the float64 oracle's
dense definition ("attention_kernels.py" section 2 ``_mask``, section 3
``flash_forward``'s ``q_start``).  Same bars as the square case: O max-abs 1e-2
(plus the bf16 output's half-ulp), LSE max-abs 2e-3, gradients 2e-2 relative
Frobenius; keys that no query sees must get exactly zero dK and dV."""
import numpy as np
import pytest
import torch

from oracle import attention_dense, attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, LSE_MAX_ABS, f64, max_abs, o_within_bar, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(B, H, Nq, Nk, d, seed):
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, _, _, do = make_attention_inputs(B, H, Nq, d, seed, "cuda")
    _, k, v, _ = make_attention_inputs(B, H, Nk, d, seed + 1000, "cuda", with_do=False)
    return q, k, v, do


CASES = [
    # B, H, Nq, Nk, q_start, d, causal
    (1, 2, 300, 1000, 700, 128, True),    # chunked prefill: the last 300 positions
    (2, 2, 4, 3000, 2996, 64, True),      # multi-token decoding with a causal mask
    (1, 3, 200, 1000, 0, 128, True),      # queries at the start: keys past 199 unseen
    (1, 2, 333, 777, 0, 128, False),      # cross-attention
    (1, 2, 500, 200, 0, 64, True),        # more queries than keys: rows >= 199 see all
    (2, 1, 500, 500, 37, 128, True),      # an offset that is no multiple of a tile
    (1, 1, 129, 4100, 3971, 128, True),   # ragged tiles on both axes
]


@pytest.mark.parametrize("B,H,Nq,Nk,q_start,d,causal", CASES)
def test_forward_with_query_offset(B, H, Nq, Nk, q_start, d, causal):
    from exact_attention_flash_gb300 import fa_device_status, fa_forward

    q, k, v, _ = _inputs(B, H, Nq, Nk, d, 31)
    o, lse = fa_forward(q, k, v, causal=causal, q_start=q_start, out_dtype=torch.float32)
    ob, _ = fa_forward(q, k, v, causal=causal, q_start=q_start)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v), causal=causal, q_start=q_start)
    assert max_abs(f64(o), ref_o) <= 1e-2
    assert o_within_bar(f64(ob), ref_o, "bf16") <= 0.0
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS


@pytest.mark.parametrize("B,H,Nq,Nk,q_start,d,causal", [c for c in CASES if c[2] * c[3] <= 2_000_000])
def test_backward_with_query_offset(B, H, Nq, Nk, q_start, d, causal):
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward

    q, k, v, do = _inputs(B, H, Nq, Nk, d, 32)
    o, lse = fa_forward(q, k, v, causal=causal, q_start=q_start)
    dq, dk, dv = fa_backward(q, k, v, o, lse, do, causal=causal, q_start=q_start)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=causal, q_start=q_start)
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        err = rel_fro(f64(got), r)
        assert err <= GRAD_REL_FRO, f"{name}: relative Frobenius error {err:.3e}"
    if causal:
        unseen = q_start + Nq  # keys at positions >= q_start + Nq are seen by no query
        if unseen < Nk:
            assert torch.count_nonzero(dk[:, :, unseen:]) == 0
            assert torch.count_nonzero(dv[:, :, unseen:]) == 0


def test_square_call_equals_offset_zero():
    """fa_forward with Nq = Nk and q_start = 0 is the square case, bit for bit."""
    from exact_attention_flash_gb300 import fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(1, 2, 640, 128, 33, "cuda", with_do=False)
    o1, l1 = fa_forward(q, k, v, causal=True)
    o2, l2 = fa_forward(q, k, v, causal=True, q_start=0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_offset_arguments_are_checked():
    from exact_attention_flash_gb300 import FAError, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(1, 1, 64, 64, 34, "cuda", with_do=False)
    with pytest.raises(FAError):
        fa_forward(q, k, v, causal=True, q_start=-1)
    with pytest.raises(ValueError):
        fa_forward(q, k[:, :, :, :32].contiguous(), v, causal=True)
    with pytest.raises(ValueError):
        fa_forward(q, k, v, out=torch.empty(1, 1, 63, 64, device="cuda", dtype=torch.bfloat16))
