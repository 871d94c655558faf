"""Pins of the oracle's block-wise loop and its counters ("attention_kernels.py",
sections 3, 4 and 6: ``flash_forward`` and ``flash_backward`` with ``stats``, and
``io_flash``).

The loop's results are pinned to the dense definition at float64 rounding for
even and uneven blocks.  Its counters are pinned to closed forms (square causal
blocks: n(n+1)/2 computed, n(n-1)/2 skipped) and to an element-wise brute force
that never runs the loop: a block is computed when any (query, key) pair in it is
visible, a row's "rescale" is a strict growth of the running maximum of its
per-block score maxima (taken from the dense score matrix), and each computed
block adds its rows times d to dQ.  ``io_flash`` is pinned to values worked out by
hand from the page's formula.
"""
import math

import numpy as np
import pytest

from oracle import (
    attention_dense,
    attention_dense_backward,
    attention_flash_blocked,
    attention_flash_blocked_backward,
    default_scale,
    io_flash,
)

BLOCKS = [(1, 1), (2, 3), (4, 4), (5, 7), (8, 2), (16, 16), (64, 128)]


def _inputs(n, d, seed):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((n, d)) for _ in range(4))


def _visible(n, causal):
    return np.tril(np.ones((n, n), dtype=bool)) if causal else np.ones((n, n), dtype=bool)


def _block_any(mask, br, bc):
    """(query block, key block) -> whether any element of the block is True."""
    n_i, n_j = -(-mask.shape[0] // br), -(-mask.shape[1] // bc)
    out = np.zeros((n_i, n_j), dtype=bool)
    for a in range(n_i):
        for b in range(n_j):
            out[a, b] = mask[a * br:(a + 1) * br, b * bc:(b + 1) * bc].any()
    return out


def _brute_rescales(q, k, br, bc, causal):
    sc = default_scale(q.shape[1], None)
    s = (q @ k.T) * sc
    vis = _visible(q.shape[0], causal)
    s = np.where(vis, s, -np.inf)
    computed = _block_any(vis, br, bc)
    total = 0
    for i in range(q.shape[0]):
        blocks = [j for j in range(computed.shape[1]) if computed[i // br, j]]
        mx = np.array([s[i, j * bc:(j + 1) * bc].max() for j in blocks])
        run = np.maximum.accumulate(mx)
        total += int(np.count_nonzero((run[1:] > run[:-1]) & np.isfinite(run[:-1])))
    return total


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", BLOCKS)
def test_blocked_forward_equals_dense(br, bc, causal):
    q, k, v, _ = _inputs(37, 8, 1)
    o, lse = attention_flash_blocked(q, k, v, br, bc, causal=causal)
    od, ld = attention_dense(q[None, None], k[None, None], v[None, None], causal=causal)
    assert np.abs(o - od[0, 0]).max() < 1e-12
    assert np.abs(lse - ld[0, 0]).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", BLOCKS)
def test_blocked_backward_equals_dense(br, bc, causal):
    q, k, v, do = _inputs(29, 8, 2)
    od, ld = attention_dense(q[None, None], k[None, None], v[None, None], causal=causal)
    grads = attention_flash_blocked_backward(q, k, v, od[0, 0], ld[0, 0], do, br, bc, causal=causal)
    ref = attention_dense_backward(q[None, None], k[None, None], v[None, None], do[None, None], causal=causal)
    for g, r in zip(grads, ref):
        assert np.abs(g - r[0, 0]).max() < 1e-11


@pytest.mark.parametrize("n_blocks,b", [(1, 4), (3, 4), (8, 16), (5, 1)])
def test_counters_closed_form_square_causal(n_blocks, b):
    n = n_blocks * b
    q, k, v, do = _inputs(n, 4, 3)
    st = {}
    o, lse = attention_flash_blocked(q, k, v, b, b, causal=True, stats=st)
    assert st.get("tiles", 0) == n_blocks * (n_blocks + 1) // 2
    assert st.get("skipped", 0) == n_blocks * (n_blocks - 1) // 2
    sb = {}
    attention_flash_blocked_backward(q, k, v, o, lse, do, b, b, causal=True, stats=sb)
    # block (i, j) with j <= i adds b rows * d
    assert sb["dq_atomic_adds"] == (n_blocks * (n_blocks + 1) // 2) * b * 4


@pytest.mark.parametrize("n", [37, 64, 100])
def test_counters_closed_form_noncausal(n):
    q, k, v, do = _inputs(n, 4, 4)
    st = {}
    o, lse = attention_flash_blocked(q, k, v, 16, 32, causal=False, stats=st)
    assert st["tiles"] == math.ceil(n / 16) * math.ceil(n / 32)
    assert st.get("skipped", 0) == 0
    sb = {}
    attention_flash_blocked_backward(q, k, v, o, lse, do, 16, 32, causal=False, stats=sb)
    assert sb["dq_atomic_adds"] == n * 4 * math.ceil(n / 32)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(2, 3), (5, 7), (8, 2), (16, 8), (3, 16)])
def test_counters_match_elementwise_brute_force(br, bc, causal):
    n, d = 45, 4
    q, k, v, do = _inputs(n, d, 5)
    st = {}
    o, lse = attention_flash_blocked(q, k, v, br, bc, causal=causal, stats=st)
    computed = _block_any(_visible(n, causal), br, bc)
    assert st.get("tiles", 0) == int(computed.sum())
    assert st.get("skipped", 0) == int(computed.size - computed.sum())
    assert st.get("rescales", 0) == _brute_rescales(q, k, br, bc, causal)
    sb = {}
    attention_flash_blocked_backward(q, k, v, o, lse, do, br, bc, causal=causal, stats=sb)
    rows = np.array([min(br, n - a * br) for a in range(computed.shape[0])])
    assert sb["dq_atomic_adds"] == int((computed.sum(axis=1) * rows).sum()) * d


def test_rescale_margin_brackets():
    q, k, v, _ = _inputs(50, 8, 6)
    counts = []
    for margin in (-np.inf, -0.5, 0.0, 0.5, np.inf):
        st = {}
        attention_flash_blocked(q, k, v, 8, 8, causal=True, stats=st, rescale_margin=margin)
        counts.append(st.get("rescales", 0))
    assert counts == sorted(counts, reverse=True)
    assert counts[-1] == 0
    # margin -inf counts every computed (row, block) after the row's first finite maximum
    vis = _visible(50, True)
    computed = _block_any(vis, 8, 8)
    every = sum(int(computed[i // 8].sum()) - 1 for i in range(50))
    assert counts[0] == every


def test_io_flash_hand_values():
    # 2 N d + 2 N d ceil(N / Br) + N
    assert io_flash(8, 2, 4) == 2 * 8 * 2 + 2 * 8 * 2 * 2 + 8 == 104
    assert io_flash(10, 3, 4) == 60 + 60 * 3 + 10 == 250
    # K and V read once: 4 N d + N
    assert io_flash(8, 2, 4, kv_cached=True) == 72
    assert io_flash(8192, 128, 128, kv_cached=True) == 4 * 8192 * 128 + 8192


def test_blocked_rejects_empty_blocks():
    q, k, v, _ = _inputs(4, 2, 7)
    with pytest.raises(ValueError):
        attention_flash_blocked(q, k, v, 0, 2)
    with pytest.raises(ValueError):
        attention_flash_blocked_backward(q, k, v, q, q[:, 0], q, 2, 0)
