"""Backward parity: the sm_103a kernels through the C ABI against the float64
oracle's dense-definition gradient on the same bf16 inputs (relative Frobenius
error of dQ, dK, dV each <= 2e-2), plus invariants that hold at any size."""
import numpy as np
import pytest
import torch

from oracle import attention_dense_backward
from tests.gpu_util import GRAD_REL_FRO, f64, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(B, H, N, d, causal, seed, mult=1.0, o_dtype=torch.bfloat16):
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, do = make_attention_inputs(B, H, N, d, seed, "cuda", qk_mult=mult)
    o, lse = fa_forward(q, k, v, causal=causal, out_dtype=o_dtype)
    dq, dk, dv = fa_backward(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    return q, k, v, do, dq, dk, dv


def _check(got, ref):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = f64(g)
        assert np.isfinite(g).all(), name
        err = rel_fro(g, r)
        assert err <= GRAD_REL_FRO, f"{name} relative Frobenius error {err:.3e}"


SMALL = [
    (1, 1, 128, 64),
    (1, 1, 256, 128),
    (2, 3, 300, 64),
    (1, 2, 515, 128),
    (2, 1, 1, 64),
    (1, 1, 129, 128),
    (1, 1, 63, 64),
    (3, 1, 640, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_backward_matches_oracle_small(shape, causal):
    B, H, N, d = shape
    q, k, v, do, dq, dk, dv = _run(B, H, N, d, causal, seed=200 + N + d)
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=causal)
    _check((dq, dk, dv), ref)


def test_backward_fp32_o_and_large_logits():
    q, k, v, do, dq, dk, dv = _run(1, 2, 384, 128, True, seed=9, mult=8.0, o_dtype=torch.float32)
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=True)
    _check((dq, dk, dv), ref)


def _invariants(dk, dv, do):
    """Rows of P sum to one: the key-sum of dK is zero and the key-sum of dV equals
    the row-sum of dO, per head."""
    dk_sum = dk.double().sum(dim=-2)
    dv_sum = dv.double().sum(dim=-2)
    do_sum = do.double().sum(dim=-2)
    scale_k = dk.double().abs().sum(dim=-2).clamp_min(1e-30)
    assert float((dk_sum.abs() / scale_k).max()) <= 2e-2
    assert float(((dv_sum - do_sum).abs() / do.double().abs().sum(dim=-2)).max()) <= 2e-2


def test_backward_causal_b4h16_n2048_d64_full():
    """Full-size causal backward (seed 1): every gradient element compared."""
    q, k, v, do, dq, dk, dv = _run(4, 16, 2048, 64, True, seed=1)
    ref = attention_dense_backward(f64(q), f64(k), f64(v), f64(do), causal=True)
    _check((dq, dk, dv), ref)
    _invariants(dk, dv, do)


def test_backward_causal_b2h16_n8192_d128_qk8_sampled_heads():
    """Full-size causal backward with Q, K x8 (seed 2): four whole heads compared
    element by element (both batches, first, middle and last heads); the dK / dV
    invariants on every head."""
    q, k, v, do, dq, dk, dv = _run(2, 16, 8192, 128, True, seed=2, mult=8.0)
    for b, h in [(0, 0), (0, 10), (1, 6), (1, 15)]:
        ref = attention_dense_backward(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h]), causal=True)
        _check((dq[b, h], dk[b, h], dv[b, h]), ref)
    _invariants(dk, dv, do)
