"""Split-KV decode parity: kernel (with its in-kernel merge) against the oracle's
split/merge decode on the same bf16 inputs, including the per-segment states."""
import numpy as np
import pytest
import torch

from oracle import attention_dense, attention_split_decode
from tests.gpu_util import LSE_MAX_ABS, O_MAX_ABS, f64, max_abs, require_gpu

pytestmark = pytest.mark.gpu

# Tighter than the O/LSE bars: decode works in fp32 end to end.
STATE_REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _decode(B, H, L, d, n_split, seed):
    from exact_attention_flash_gb300 import fa_decode, fa_device_status
    from exact_attention_flash_gb300.workloads import make_decode_inputs

    q, k, v = make_decode_inputs(B, H, L, d, seed, "cuda")
    o, lse, parts = fa_decode(q, k, v, n_split, return_partials=True)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    return q, k, v, o, lse, parts


def _check_head(q, k, v, o, lse, parts, n_split):
    ref_o, ref_l, ref_parts = attention_split_decode(f64(q), f64(k), f64(v), n_split)
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS
    assert max_abs(f64(lse), ref_l[..., 0]) <= LSE_MAX_ABS
    dense_o, _ = attention_dense(f64(q), f64(k), f64(v))
    assert max_abs(f64(o), dense_o) <= 1e-4
    got = f64(parts)
    for s, st in enumerate(ref_parts):
        m, l, ov = got[..., s, 0], got[..., s, 1], got[..., s, 2:]
        empty = np.isneginf(st.m[..., 0])
        assert np.all(np.isneginf(m[empty])) and np.all(l[empty] == 0) and np.all(ov[empty] == 0)
        ok = ~empty
        np.testing.assert_allclose(m[ok], st.m[..., 0][ok], rtol=STATE_REL, atol=1e-4)
        np.testing.assert_allclose(l[ok], st.l[..., 0][ok], rtol=STATE_REL)
        np.testing.assert_allclose(ov[ok], st.o[..., 0, :][ok], rtol=STATE_REL, atol=1e-4 * np.max(st.l))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L,n_split", [(1, 1), (7, 3), (100, 64), (1000, 7), (4097, 64), (33, 40), (2048, 1)])
def test_decode_matches_oracle_small(L, n_split, d):
    q, k, v, o, lse, parts = _decode(2, 3, L, d, n_split, seed=L + d)
    _check_head(q, k, v, o, lse, parts, n_split)


def test_decode_b16h32_l32768_d128_s64_all_heads():
    """Full-size decode (seed 4): every one of the 512 (batch, head) pairs compared
    with the oracle's split-and-merge decode: O, LSE and all 64 segment states, and
    O against the dense definition.  The oracle runs one batch (32 heads) at a time."""
    q, k, v, o, lse, parts = _decode(16, 32, 32768, 128, 64, seed=4)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for b in range(16):
        _check_head(q[b], k[b], v[b], o[b], lse[b], parts[b], 64)


def test_decode_twice_reuses_workspace():
    """The arrival counters are cleared per call: a second call on the same
    workspace gives the same result."""
    from exact_attention_flash_gb300 import decode_workspace_bytes, fa_decode
    from exact_attention_flash_gb300.workloads import make_decode_inputs

    q, k, v = make_decode_inputs(2, 4, 3000, 128, 11, "cuda")
    ws = torch.empty(decode_workspace_bytes(2, 4, 128, 16), device="cuda", dtype=torch.uint8)
    o1, l1 = fa_decode(q, k, v, 16, workspace=ws)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = fa_decode(q, k, v, 16, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
