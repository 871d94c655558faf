"""Parity at the extremes of the sizes the kernels take: a long ragged sequence
(the forward's grid along N and its last, partial query tile), thousands of heads
with a single ragged key tile each (the backward's grid along batch*head), more
heads than a grid's y or z dimension holds, and a long ragged decode context.
Same bars as the other parity tests."""
import numpy as np
import pytest
import torch

from oracle import attention_dense_backward, attention_dense_rows, attention_split_decode
from tests.gpu_util import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, f64, max_abs, o_within_bar, rel_fro, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("causal", [False, True])
def test_forward_long_ragged_sequence_sampled_rows(causal):
    """B=1, H=2, N=65613 (256 full query blocks plus a ragged one), d=128: sampled
    rows, including both ends of the tile boundaries and the last row."""
    from exact_attention_flash_gb300 import fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    N = 65613
    q, k, v, _ = make_attention_inputs(1, 2, N, 128, 11, "cuda", with_do=False)
    o, lse = fa_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = [0, 1, 127, 128, 255, 256, 32768, 65535, 65536, 65600, N - 1]
    for h in range(2):
        ref_o, ref_l = attention_dense_rows(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), rows, causal=causal)
        go, gl = f64(o[0, h, rows]), f64(lse[0, h, rows])
        assert o_within_bar(go, ref_o, "bf16") <= 0.0, f"O error {max_abs(go, ref_o):.3e}"
        assert max_abs(gl, ref_l) <= LSE_MAX_ABS


@pytest.mark.parametrize("causal", [False, True])
def test_backward_4096_heads_of_one_ragged_tile(causal):
    """B=64, H=64, N=65, d=64: 4096 heads, each a single partial key tile and two
    query blocks (one of a single row); sampled heads against the dense gradient,
    every gradient finite."""
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, do = make_attention_inputs(64, 64, 65, 64, 12, "cuda")
    o, lse = fa_forward(q, k, v, causal=causal)
    dq, dk, dv = fa_backward(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    for g in (dq, dk, dv):
        assert torch.isfinite(g).all()
    for b, h in [(0, 0), (17, 40), (63, 63)]:
        ref = attention_dense_backward(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h]), causal=causal)
        for name, got, r in zip(("dQ", "dK", "dV"), (dq[b, h], dk[b, h], dv[b, h]), ref):
            err = rel_fro(f64(got), r)
            assert err <= GRAD_REL_FRO, f"{name} of ({b}, {h}): relative Frobenius error {err:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_more_heads_than_a_grid_dimension(causal):
    """B=70, H=1000: 70 000 heads (more than 65535, the limit of a grid's y and z
    dimensions) of N=20, d=64, forward and backward.  Heads on both sides of 65535
    against the oracle, every output finite."""
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs
    from oracle import attention_dense

    q, k, v, do = make_attention_inputs(70, 1000, 20, 64, 14, "cuda")
    o, lse = fa_forward(q, k, v, causal=causal)
    dq, dk, dv = fa_backward(q, k, v, o, lse, do, causal=causal, grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    for flat in (0, 4321, 65534, 65535, 65536, 69999):
        b, h = divmod(flat, 1000)
        ref_o, ref_l = attention_dense(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), causal=causal)
        assert o_within_bar(f64(o[b, h]), ref_o, "bf16") <= 0.0
        assert max_abs(f64(lse[b, h]), ref_l) <= LSE_MAX_ABS
        ref = attention_dense_backward(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(do[b, h]), causal=causal)
        for name, got, r in zip(("dQ", "dK", "dV"), (dq[b, h], dk[b, h], dv[b, h]), ref):
            err = rel_fro(f64(got), r)
            assert err <= GRAD_REL_FRO, f"{name} of head {flat}: relative Frobenius error {err:.3e}"


def test_decode_long_ragged_context():
    """B=1, H=2, L=300001 keys in 128 splits (uneven segments), d=128."""
    from exact_attention_flash_gb300 import fa_decode, fa_device_status
    from exact_attention_flash_gb300.workloads import make_decode_inputs

    q, k, v = make_decode_inputs(1, 2, 300001, 128, 13, "cuda")
    o, lse = fa_decode(q, k, v, 128)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l, _ = attention_split_decode(f64(q), f64(k), f64(v), 128)
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS
    assert max_abs(f64(lse), ref_l[..., 0]) <= LSE_MAX_ABS
    assert np.isfinite(f64(o)).all()


def test_forward_concurrent_streams_and_slot_reuse():
    """The persistent forward claims work items from one of a rotating set of
    scheduling slots.  Launches overlapping on four streams (different inputs)
    must each be complete and correct, and 130 launches in a row (every slot
    reused) must keep returning the same result."""
    from exact_attention_flash_gb300 import fa_device_status, fa_forward
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    inputs = [make_attention_inputs(1, 4, 1000, 128, 40 + i, "cuda", with_do=False)[:3] for i in range(4)]
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = [None] * 4
    torch.cuda.synchronize()
    for _ in range(3):
        for i, (st, (q, k, v)) in enumerate(zip(streams, inputs)):
            with torch.cuda.stream(st):
                outs[i] = fa_forward(q, k, v, causal=bool(i & 1), stream=st)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    for i, (q, k, v) in enumerate(inputs):
        o, lse = outs[i]
        rows = [0, 1, 255, 256, 511, 512, 999]
        for h in (0, 3):
            ref_o, ref_l = attention_dense_rows(f64(q[0, h]), f64(k[0, h]), f64(v[0, h]), rows, causal=bool(i & 1))
            assert o_within_bar(f64(o[0, h, rows]), ref_o, "bf16") <= 0.0
            assert max_abs(f64(lse[0, h, rows]), ref_l) <= LSE_MAX_ABS
    q, k, v = inputs[0]
    o0, l0 = fa_forward(q, k, v)
    o, lse = torch.empty_like(o0), torch.empty_like(l0)
    for _ in range(130):
        fa_forward(q, k, v, out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    assert torch.equal(o, o0) and torch.equal(lse, l0)
