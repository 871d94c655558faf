"""The kernels' counters of the page's ``stats`` ("attention_kernels.py" sections 3
and 4: "tiles", "skipped", "rescales", "dq_atomic_adds"; enabled with
``fa_set_stats``) against the oracle's block-wise loop run with the kernels'
blocks (forward 128 x 128, backward 64 x 128), one head at a time.

Tiles, skipped tiles and dQ additions depend only on the shapes and are compared
exactly.  A rescale is a floating-point decision (did a row's running maximum
grow?), taken by the kernel on fp32 tensor-core scores and by the oracle in
float64, so the kernel's count is checked to lie between the oracle's counts
with a growth threshold of +1e-3 and -1e-3 (scaled score units; the fp32 score
error at d = 128 is near 1e-5 here).
"""
import numpy as np
import pytest
import torch

from oracle import attention_dense, attention_flash_blocked, attention_flash_blocked_backward
from tests.gpu_util import f64, require_gpu

pytestmark = pytest.mark.gpu

MARGIN = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _oracle_forward_counts(q, k, v, causal):
    B, H = q.shape[:2]
    tiles = skipped = lo = hi = 0
    for b in range(B):
        for h in range(H):
            st, st_lo, st_hi = {}, {}, {}
            attention_flash_blocked(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), 128, 128, causal=causal, stats=st)
            attention_flash_blocked(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), 128, 128, causal=causal,
                                    stats=st_lo, rescale_margin=MARGIN)
            attention_flash_blocked(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), 128, 128, causal=causal,
                                    stats=st_hi, rescale_margin=-MARGIN)
            tiles += st.get("tiles", 0)
            skipped += st.get("skipped", 0)
            lo += st_lo.get("rescales", 0)
            hi += st_hi.get("rescales", 0)
    return tiles, skipped, lo, hi


@pytest.mark.parametrize("B,H,N,d,causal,qk", [
    (2, 3, 700, 128, True, 1.0),
    (2, 3, 700, 128, False, 1.0),
    (1, 2, 1000, 64, True, 1.0),
    (1, 1, 1, 128, True, 1.0),
    (1, 1, 4096, 128, True, 8.0),
])
def test_forward_counters_match_oracle(B, H, N, d, causal, qk):
    from exact_attention_flash_gb300 import fa_device_status, fa_forward, stats_counters
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(B, H, N, d, 21, "cuda", with_do=False, qk_mult=qk)
    with stats_counters() as c:
        fa_forward(q, k, v, causal=causal)
        torch.cuda.synchronize()
    assert fa_device_status() == 0
    tiles, skipped, resc, dq_adds = (int(x) for x in c.cpu())
    o_tiles, o_skipped, lo, hi = _oracle_forward_counts(q, k, v, causal)
    assert tiles == o_tiles
    assert skipped == o_skipped
    assert lo <= resc <= hi, f"rescales {resc} outside [{lo}, {hi}]"
    assert dq_adds == 0


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 700, 128, True), (1, 2, 1000, 64, False), (1, 1, 65, 128, True)])
def test_backward_dq_additions_match_oracle(B, H, N, d, causal):
    from exact_attention_flash_gb300 import fa_backward, fa_device_status, fa_forward, stats_counters
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, do = make_attention_inputs(B, H, N, d, 22, "cuda")
    o, lse = fa_forward(q, k, v, causal=causal)
    with stats_counters() as c:
        fa_backward(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
    assert fa_device_status() == 0
    counts = [int(x) for x in c.cpu()]
    st = {}
    qh, kh, vh, doh = (f64(t[0, 0]) for t in (q, k, v, do))
    oh, lh = attention_dense(qh[None, None], kh[None, None], vh[None, None], causal=causal)
    attention_flash_blocked_backward(qh, kh, vh, oh[0, 0], lh[0, 0], doh, 64, 128, causal=causal, stats=st)
    # the count depends on the shapes only: one head's count times B * H
    assert counts[3] == st["dq_atomic_adds"] * B * H
    assert counts[:3] == [0, 0, 0]


def test_counters_accumulate_and_stop():
    from exact_attention_flash_gb300 import fa_forward, fa_set_stats
    from exact_attention_flash_gb300.workloads import make_attention_inputs

    q, k, v, _ = make_attention_inputs(1, 2, 512, 128, 23, "cuda", with_do=False)
    c = torch.zeros(4, dtype=torch.int64, device="cuda")
    fa_set_stats(c)
    try:
        fa_forward(q, k, v, causal=True)
        fa_forward(q, k, v, causal=True)
    finally:
        fa_set_stats(None)
    fa_forward(q, k, v, causal=True)  # not counted
    torch.cuda.synchronize()
    # 4 query tiles of 128 rows: 1 + 2 + 3 + 4 key tiles computed, 3 + 2 + 1 skipped; 2 heads; 2 calls
    assert int(c[0]) == 2 * 2 * 10
    assert int(c[1]) == 2 * 2 * 6
    with pytest.raises(ValueError):
        fa_set_stats(torch.zeros(4, dtype=torch.int32, device="cuda"))
