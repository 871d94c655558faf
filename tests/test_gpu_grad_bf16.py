"""Backward with bf16 gradients (grad_dtype = bf16).

Every product still accumulates in fp32. Only the final dQ, dK and dV are rounded
to bf16. So:
- Against the float64 oracle ("attention_kernels.py" section 4 ``flash_backward``)
  the usual bar holds: relative Frobenius error <= 2e-2.
- dK and dV must equal, bit for bit, the bf16 rounding of the same call's fp32
  gradients. The tensor-core accumulation order is fixed, so the fp32 values are
  the same in both calls.
- dQ is summed over key tiles by fp32 reductions whose order varies from call to
  call, so the two calls' fp32 sums differ in their last bits (more where the
  partial sums cancel). The bf16 call leaves its fp32 accumulator in the workspace
  (after the bias tiles, at a 256-byte boundary, as the header states). dQ must be
  that accumulator rounded to bf16, bit for bit, and the accumulator must match the
  fp32 call's dQ to 1e-4 in relative Frobenius norm (bf16 rounding alone is 2^-9).
- Keys that no query sees (a query offset) get exactly zero gradients.
"""
import pytest
import torch

from oracle import attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, f64, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _both(B, H, Nq, Nk, d, causal, seed, q_start=0, mult=1.0):
    from exact_attention_flash_gb300 import backward_workspace_bytes, fa_backward, fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, do = make_attention_inputs(B, H, Nq, d, seed, "cuda", qk_mult=mult)
    if Nk != Nq:
        _, k, v, _ = make_attention_inputs(B, H, Nk, d, seed + 1000, "cuda", qk_mult=mult, with_do=False)
    o, lse = fa_forward(q, k, v, causal=causal, q_start=q_start)
    g32 = fa_backward(q, k, v, o, lse, do, causal=causal, q_start=q_start)
    ws = torch.empty(backward_workspace_bytes(B, H, Nq, d, torch.bfloat16), device="cuda", dtype=torch.uint8)
    g16 = fa_backward(q, k, v, o, lse, do, causal=causal, q_start=q_start, grad_dtype=torch.bfloat16, workspace=ws)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    assert all(g.dtype == torch.bfloat16 for g in g16)
    off = -(-backward_workspace_bytes(B, H, Nq, d) // 256) * 256  # the bias tiles, rounded up to 256 bytes
    acc = ws[off: off + B * H * Nq * d * 4].view(torch.float32).view(B, H, Nq, d)
    return (q, k, v, do), g32, g16, acc


def _consistent(g32, g16, acc):
    dq32, dk32, dv32 = g32
    dq16, dk16, dv16 = g16
    assert torch.equal(dk16, dk32.to(torch.bfloat16))
    assert torch.equal(dv16, dv32.to(torch.bfloat16))
    assert torch.equal(dq16, acc.to(torch.bfloat16))
    assert rel_fro(f64(acc), f64(dq32)) <= 1e-4


CASES = [
    # B, H, N, d, causal
    (1, 1, 128, 64, False),
    (2, 3, 300, 64, True),
    (1, 2, 515, 128, True),
    (1, 1, 129, 128, False),
    (2, 1, 1, 64, True),
    (3, 1, 640, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", CASES)
def test_bf16_gradients_match_oracle(B, H, N, d, causal):
    (q, k, v, do), g32, g16, acc = _both(B, H, N, N, d, causal, seed=400 + N + d)
    _consistent(g32, g16, acc)
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=causal)
    for name, got, r in zip(("dQ", "dK", "dV"), g16, ref):
        err = rel_fro(f64(got), r)
        assert err <= GRAD_REL_FRO, f"{name}: relative Frobenius error {err:.3e}"


def test_bf16_gradients_with_query_offset_and_unseen_keys():
    B, H, Nq, Nk, q_start, d = 1, 2, 200, 1000, 0, 128   # keys past position 199 are seen by no query
    (q, k, v, do), g32, g16, acc = _both(B, H, Nq, Nk, d, True, seed=41, q_start=q_start)
    _consistent(g32, g16, acc)
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=True, q_start=q_start)
    for name, got, r in zip(("dQ", "dK", "dV"), g16, ref):
        assert rel_fro(f64(got), r) <= GRAD_REL_FRO, name
    assert torch.count_nonzero(g16[1][:, :, Nq:]) == 0
    assert torch.count_nonzero(g16[2][:, :, Nq:]) == 0


def test_bf16_gradients_full_size_b2h16_n8192_d128_qk8():
    """The causal N = 8192, d = 128 workload (Q, K x8, seed 2): consistency with the
    fp32 gradients everywhere, and two heads against the oracle element by element."""
    (q, k, v, do), g32, g16, acc = _both(2, 16, 8192, 8192, 128, True, seed=2, mult=8.0)
    _consistent(g32, g16, acc)
    for b, h in [(0, 5), (1, 14)]:
        ref = attention_dense_backward(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h]), causal=True)
        for name, got, r in zip(("dQ", "dK", "dV"), (g[b, h] for g in g16), ref):
            assert rel_fro(f64(got), r) <= GRAD_REL_FRO, name


def test_bf16_gradients_reject_wrong_buffers():
    from exact_attention_flash_gb300 import backward_workspace_bytes, fa_backward, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, do = make_attention_inputs(1, 1, 64, 64, 3, "cuda")
    o, lse = fa_forward(q, k, v)
    with pytest.raises(ValueError):  # fp32 buffers for bf16 gradients
        fa_backward(q, k, v, o, lse, do, grad_dtype=torch.bfloat16, dq=torch.empty_like(q, dtype=torch.float32))
    with pytest.raises(ValueError):
        fa_backward(q, k, v, o, lse, do, grad_dtype=torch.float16)
    small = torch.empty(backward_workspace_bytes(1, 1, 64, 64), device="cuda", dtype=torch.uint8)
    with pytest.raises(RuntimeError):  # the fp32-gradient workspace has no room for the dQ accumulator
        fa_backward(q, k, v, o, lse, do, grad_dtype=torch.bfloat16, workspace=small)
