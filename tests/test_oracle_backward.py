"""Pins for the oracle's gradient paths (dense definition and row-wise tiled).

Central finite differences of loss = sum(O * dO) ("lab.py" ``finite_difference``,
h = 1e-5, atol 2e-8, rtol 2e-6), float64 autograd through a softmax written with
torch's own library routine ("model.py" verify() compares against autograd), and
the invariants that follow from rows of P summing to one.
"""
import math

import numpy as np
import pytest
import torch

from oracle import (
    attention_dense,
    attention_dense_backward,
    attention_tiled_rowwise,
    attention_tiled_rowwise_backward,
)


def _finite_difference(q, k, v, do, causal, h=1e-5):
    grads = []
    for arr in (q, k, v):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            plus = np.sum(attention_dense(q, k, v, causal=causal)[0] * do)
            arr[idx] = old - h
            minus = np.sum(attention_dense(q, k, v, causal=causal)[0] * do)
            arr[idx] = old
            g[idx] = (plus - minus) / (2 * h)
        grads.append(g)
    return grads


def _autograd(q, k, v, do, causal):
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    s = tq @ tk.transpose(-1, -2) / math.sqrt(q.shape[-1])
    if causal:
        n = q.shape[-2]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    out = torch.softmax(s, dim=-1) @ tv
    (out * torch.tensor(do)).sum().backward()
    return [t.grad.numpy() for t in (tq, tk, tv)]


@pytest.mark.parametrize("n", [1, 2, 5, 7, 8])
@pytest.mark.parametrize("d", [3, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(n, d, causal):
    rng = np.random.default_rng(7 + 10 * n + d)
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    numerical = _finite_difference(q.copy(), k.copy(), v.copy(), do, causal)
    dense = attention_dense_backward(q, k, v, do, causal=causal)
    out, lse = attention_tiled_rowwise(q, k, v, 3, causal=causal)
    tiled = attention_tiled_rowwise_backward(q, k, v, out, lse, do, 3, causal=causal)
    for a, b, c in zip(dense, tiled, numerical):
        np.testing.assert_allclose(a, c, atol=2e-8, rtol=2e-6)
        np.testing.assert_allclose(b, c, atol=2e-8, rtol=2e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_float64_autograd(causal):
    rng = np.random.default_rng(21)
    q, k, v, do = (rng.normal(size=(2, 3, 13, 8)) for _ in range(4))
    want = _autograd(q, k, v, do, causal)
    got = attention_dense_backward(q, k, v, do, causal=causal)
    for a, b in zip(got, want):
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=1e-11)
    for bb in range(2):
        for hh in range(3):
            out, lse = attention_tiled_rowwise(q[bb, hh], k[bb, hh], v[bb, hh], 4, causal=causal)
            tiled = attention_tiled_rowwise_backward(q[bb, hh], k[bb, hh], v[bb, hh], out, lse, do[bb, hh], 4, causal=causal)
            for a, b in zip(tiled, want):
                np.testing.assert_allclose(a, b[bb, hh], atol=1e-12, rtol=1e-11)


@pytest.mark.parametrize("block", [1, 2, 3, 5, 16])
def test_tiled_backward_is_block_size_invariant(block):
    rng = np.random.default_rng(31)
    q, k, v, do = (rng.normal(size=(11, 4)) for _ in range(4))
    for causal in (False, True):
        ref = attention_dense_backward(q, k, v, do, causal=causal)
        out, lse = attention_tiled_rowwise(q, k, v, block, causal=causal)
        got = attention_tiled_rowwise_backward(q, k, v, out, lse, do, block, causal=causal)
        for a, b in zip(got, ref):
            np.testing.assert_allclose(a, b, atol=1e-12, rtol=1e-12)


def test_gradient_invariants():
    """Rows of P sum to one, so rows of dS sum to zero: the key-sum of dK is 0 and
    the key-sum of dV equals the row-sum of dO (causal or not)."""
    rng = np.random.default_rng(41)
    q, k, v, do = (rng.normal(size=(2, 2, 19, 8)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = attention_dense_backward(q, k, v, do, causal=causal)
        np.testing.assert_allclose(dk.sum(axis=-2), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(axis=-2), do.sum(axis=-2), atol=1e-12)
