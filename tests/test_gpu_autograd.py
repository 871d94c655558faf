"""flash_attention: fa_forward and fa_backward as one autograd node.

The gradients that loss.backward() leaves in q.grad, k.grad and v.grad must be the
library's bf16 gradients:
- dK and dV equal to a direct fa_backward(..., grad_dtype=bf16) call, bit for bit;
- dQ, whose fp32 reductions vary in order, close to that call's;
- all three within the usual 2e-2 relative Frobenius bar of the float64 oracle
  ("attention_kernels.py" section 4 ``flash_backward``).
"""
import pytest
import torch

from oracle import attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, f64, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("B,H,Nq,Nk,q_start,d,causal", [(2, 2, 300, 300, 0, 64, True), (1, 3, 200, 640, 440, 128, True),
                                                          (1, 2, 257, 257, 0, 128, False)])
def test_autograd_gradients_are_the_library_gradients(B, H, Nq, Nk, q_start, d, causal):
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward, flash_attention
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, _, _, do = make_attention_inputs(B, H, Nq, d, 60, "cuda")
    _, k, v, _ = make_attention_inputs(B, H, Nk, d, 61, "cuda", with_do=False)
    qg, kg, vg = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = flash_attention(qg, kg, vg, causal=causal, q_start=q_start)
    (o.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    assert qg.grad.dtype == torch.bfloat16 and kg.grad.shape == k.shape
    o_ref, lse = fa_forward(q, k, v, causal=causal, q_start=q_start)
    assert torch.equal(o.detach(), o_ref)
    dq, dk, dv = fa_backward(q, k, v, o_ref, lse, do, causal=causal, q_start=q_start, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(kg.grad, dk) and torch.equal(vg.grad, dv)
    assert rel_fro(f64(qg.grad), f64(dq)) <= 1e-2
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=causal, q_start=q_start)
    for name, got, r in zip(("dQ", "dK", "dV"), (qg.grad, kg.grad, vg.grad), ref):
        assert rel_fro(f64(got), r) <= GRAD_REL_FRO, name
