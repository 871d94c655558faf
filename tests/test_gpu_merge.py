"""fa_merge_states and the automatic decode split count.

The merge is compared with the oracle's ``merge_states`` ("attention_kernels.py"
section 1) applied to the states (m = LSE, l = 1, o = O) of the same inputs
(l = 0, o = 0 where LSE = -inf, the empty state).  The arithmetic is fp32, so the
bar is 2e-6 relative to the largest |O| plus, for a bf16 output, bf16's half-ulp.
End to end, attention over keys held in two pieces (two fa_forward_qk calls, or
two fa_decode calls) merged by fa_merge_states must meet the usual bars against
the dense oracle over all keys.
"""
import numpy as np
import pytest
import torch

from oracle import SoftmaxState, attention_dense, merge_states
from tests.gpu_util import LSE_MAX_ABS, O_MAX_ABS, bf16_half_ulp, f64, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _oracle_merge(o_a, l_a, o_b, l_b):
    def state(o, l):
        empty = np.isneginf(l)
        return SoftmaxState(np.where(empty, -np.inf, l), np.where(empty, 0.0, 1.0), np.where(empty[..., None], 0.0, o))

    s = merge_states(state(o_a, l_a), state(o_b, l_b))
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(s.l[..., None] > 0, s.o / np.where(s.l > 0, s.l, 1.0)[..., None], 0.0)
        lse = np.where(s.l > 0, s.m + np.log(np.where(s.l > 0, s.l, 1.0)), -np.inf)
    return o, lse


def _random_results(shape, d, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    o_a = torch.randn(shape + (d,), generator=g, device="cuda").to(dtype)
    o_b = torch.randn(shape + (d,), generator=g, device="cuda").to(dtype)
    l_a = torch.randn(shape, generator=g, device="cuda") * 3
    l_b = torch.randn(shape, generator=g, device="cuda") * 3
    flat_a, flat_b = l_a.view(-1), l_b.view(-1)
    n = flat_a.numel()
    flat_a[0: n: 7] = -torch.inf                # empty runs on one side
    flat_b[3: n: 11] = -torch.inf               # on the other, and both where the strides meet
    flat_b[1: n: 13] = flat_a[1: n: 13]         # equal maxima
    flat_b[2: n: 17] = flat_a[2: n: 17] + 100.  # one side dominates completely
    return o_a, l_a, o_b, l_b


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape,d", [((2, 3, 257), 128), ((1, 1, 1), 64), ((4, 1000), 64), ((3, 5), 12)])
def test_merge_matches_oracle(shape, d, dtype):
    from exact_attention_flash_gb300 import fa_merge_states

    o_a, l_a, o_b, l_b = _random_results(shape, d, dtype, 51)
    o, lse = fa_merge_states(o_a, l_a, o_b, l_b)
    torch.cuda.synchronize()
    ref_o, ref_l = _oracle_merge(f64(o_a), f64(l_a), f64(o_b), f64(l_b))
    got_l = f64(lse)
    assert np.array_equal(np.isneginf(got_l), np.isneginf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.abs(got_l[fin] - ref_l[fin]).max() <= 2e-6 * max(1.0, np.abs(ref_l[fin]).max())
    tol = 2e-6 * np.abs(ref_o).max()
    if dtype == torch.float32:
        assert max_abs(f64(o), ref_o) <= tol
    else:
        assert np.max(np.abs(f64(o) - ref_o) - (tol + bf16_half_ulp(ref_o))) <= 0.0


def test_merge_in_place_and_identity():
    from exact_attention_flash_gb300 import fa_merge_states

    o_a, l_a, o_b, l_b = _random_results((2, 300), 128, torch.float32, 52)
    ref = fa_merge_states(o_a, l_a, o_b, l_b)
    ref = (ref[0].clone(), ref[1].clone())
    fa_merge_states(o_a, l_a, o_b, l_b, out=o_a, lse=l_a)
    torch.cuda.synchronize()
    assert torch.equal(o_a, ref[0]) and torch.equal(l_a, ref[1])
    # merging with the empty result leaves a result unchanged
    empty_l = torch.full_like(l_b, -torch.inf)
    o, lse = fa_merge_states(o_b, l_b, torch.zeros_like(o_b), empty_l)
    torch.cuda.synchronize()
    assert torch.equal(lse, l_b)
    fin = torch.isfinite(l_b)
    assert torch.equal(o[fin], o_b[fin])


@pytest.mark.parametrize("Nk,cut,d", [(1000, 333, 128), (4096, 2048, 64), (257, 1, 128)])
def test_attention_over_two_key_pieces(Nk, cut, d):
    from exact_attention_flash_gb300 import fa_device_status, fa_forward, fa_merge_states
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, _, _, _ = make_attention_inputs(1, 2, 300, d, 53, "cuda", with_do=False)
    _, k, v, _ = make_attention_inputs(1, 2, Nk, d, 54, "cuda", with_do=False)
    o_a, l_a = fa_forward(q, k[:, :, :cut].contiguous(), v[:, :, :cut].contiguous(), out_dtype=torch.float32)
    o_b, l_b = fa_forward(q, k[:, :, cut:].contiguous(), v[:, :, cut:].contiguous(), out_dtype=torch.float32)
    o, lse = fa_merge_states(o_a, l_a, o_b, l_b)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v))
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS


def test_decode_over_two_key_pieces_and_auto_split():
    from exact_attention_flash_gb300 import decode_auto_split, fa_decode, fa_device_status, fa_merge_states
    from exact_attention_flash_gb300.workloads import make_decode_inputs

    q, k, v = make_decode_inputs(2, 4, 20000, 128, 55, "cuda")
    a = fa_decode(q, k[:, :, :7000].contiguous(), v[:, :, :7000].contiguous())
    b = fa_decode(q, k[:, :, 7000:].contiguous(), v[:, :, 7000:].contiguous())
    # decode's LSE is [B, H]; as merge input it is the [B, H, 1] of the one query row
    o, lse = fa_merge_states(a[0], a[1].unsqueeze(-1), b[0], b[1].unsqueeze(-1))
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v))
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS
    # the documented rule: ceil(4 SMs / (B H)), at least 8, at most L / 512 (at least 1)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, H, L in ((16, 32, 32768), (1, 8, 131072), (4, 8, 8192), (64, 32, 4096), (1, 1, 65536), (1, 1, 100)):
        expect = min(max(-(-4 * sms // (B * H)), 8), max(L // 512, 1))
        assert decode_auto_split(B, H, L) == expect


def test_merge_rejects_mismatched_inputs():
    from exact_attention_flash_gb300 import fa_merge_states

    o = torch.zeros(2, 8, device="cuda")
    l = torch.zeros(2, device="cuda")
    with pytest.raises(ValueError):
        fa_merge_states(o, l, o.to(torch.bfloat16), l)
    with pytest.raises(ValueError):
        fa_merge_states(o, l, o, torch.zeros(3, device="cuda"))
