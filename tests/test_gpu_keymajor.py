"""Parity of the forward in the first algorithm's key-major loop order
(fa_forward_keymajor; "flash_attention_numpy.py" ``flash_attention_tier1`` with
the scale and causal mask of "attention_kernels.py" section 3) with the float64
oracle's dense definition, at the forward's bars: O max-abs 1e-2 (plus bf16's
half-ulp for a bf16 output), LSE max-abs 2e-3."""
import pytest
import torch

from oracle import attention_dense
from tests.gpu_util import LSE_MAX_ABS, f64, max_abs, o_within_bar, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 300, 128, True),
    (2, 1, 257, 64, False),
    (1, 1, 1, 128, True),
    (1, 3, 1000, 64, True),
    (1, 1, 640, 128, False),
])
def test_keymajor_forward_matches_oracle(B, H, N, d, causal):
    from exact_attention_flash_gb300 import fa_device_status, fa_forward_keymajor
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(B, H, N, d, 61, "cuda", with_do=False)
    o32, lse = fa_forward_keymajor(q, k, v, causal=causal, out_dtype=torch.float32)
    o16, _ = fa_forward_keymajor(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v), causal=causal)
    assert max_abs(f64(o32), ref_o) <= 1e-2
    assert o_within_bar(f64(o16), ref_o, "bf16") <= 0.0
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS


def test_keymajor_large_logits():
    """Q and K x8 (the bench workload's stress): every visit repairs a growing max."""
    from exact_attention_flash_gb300 import fa_device_status, fa_forward_keymajor
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(1, 2, 700, 128, 62, "cuda", with_do=False, qk_mult=8.0)
    o, lse = fa_forward_keymajor(q, k, v, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v), causal=True)
    assert max_abs(f64(o), ref_o) <= 1e-2
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS
