"""Pins of the oracle's general query offset: queries at absolute positions
q_start .. q_start + Nq - 1 against Nk keys, key j visible to query i iff
j <= q_start + i ("attention_kernels.py" section 2 ``_mask`` and section 3
``flash_forward``'s ``q_start``).

Each pin ties the offset case to something computed without it: a query block
taken from the end of a square causal problem equals the square problem's rows
(the pinned q_start = 0 definition), a softmax over each row's visible prefix by
SciPy, the all-visible limit equal to non-causal attention, and the gradients
against central finite differences and against the square problem with dO zero
on the rows the block leaves out.
"""
import numpy as np
import pytest
import scipy.special

from oracle import attention_dense, attention_dense_backward


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("nk,nq", [(9, 3), (16, 16), (7, 1), (20, 5)])
def test_block_from_the_end_equals_square_causal_rows(nk, nq):
    q_full, k, v = _rand((1, 2, nk, 4), 1), _rand((1, 2, nk, 4), 2), _rand((1, 2, nk, 4), 3)
    q_start = nk - nq
    o, lse = attention_dense(q_full[:, :, q_start:], k, v, causal=True, q_start=q_start)
    o_full, lse_full = attention_dense(q_full, k, v, causal=True)
    assert np.abs(o - o_full[:, :, q_start:]).max() < 1e-13
    assert np.abs(lse - lse_full[:, :, q_start:]).max() < 1e-13


@pytest.mark.parametrize("nq,nk,q_start", [(4, 11, 3), (5, 5, 0), (3, 6, 10), (6, 2, 0)])
def test_rows_are_softmax_over_the_visible_prefix(nq, nk, q_start):
    q, k, v = _rand((1, 1, nq, 3), 4), _rand((1, 1, nk, 3), 5), _rand((1, 1, nk, 3), 6)
    o, lse = attention_dense(q, k, v, causal=True, q_start=q_start)
    sc = 1.0 / np.sqrt(3)
    for i in range(nq):
        last = min(nk - 1, q_start + i)
        s = (k[0, 0, : last + 1] @ q[0, 0, i]) * sc
        assert abs(lse[0, 0, i] - scipy.special.logsumexp(s)) < 1e-13
        assert np.abs(o[0, 0, i] - scipy.special.softmax(s) @ v[0, 0, : last + 1]).max() < 1e-13


def test_all_keys_visible_equals_non_causal():
    q, k, v = _rand((2, 1, 5, 4), 7), _rand((2, 1, 8, 4), 8), _rand((2, 1, 8, 4), 9)
    o_c, l_c = attention_dense(q, k, v, causal=True, q_start=7)
    o_n, l_n = attention_dense(q, k, v, causal=False)
    assert np.abs(o_c - o_n).max() < 1e-13 and np.abs(l_c - l_n).max() < 1e-13


@pytest.mark.parametrize("nq,nk,q_start", [(3, 7, 4), (2, 5, 1), (4, 4, 0)])
def test_backward_against_finite_differences(nq, nk, q_start):
    q, k, v, do = _rand((nq, 3), 10), _rand((nk, 3), 11), _rand((nk, 3), 12), _rand((nq, 3), 13)
    dq, dk, dv = (g[0, 0] for g in attention_dense_backward(q[None, None], k[None, None], v[None, None],
                                                            do[None, None], causal=True, q_start=q_start))

    def loss():
        return np.sum(attention_dense(q[None, None], k[None, None], v[None, None], causal=True,
                                      q_start=q_start)[0][0, 0] * do)

    h = 1e-5
    for arr, g in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            plus = loss()
            arr[idx] = old - h
            minus = loss()
            arr[idx] = old
            fd[idx] = (plus - minus) / (2 * h)
        np.testing.assert_allclose(g, fd, atol=2e-8, rtol=2e-6)


def test_backward_block_equals_square_problem_with_zero_do_elsewhere():
    nk, nq = 12, 5
    q_start = nk - nq
    q_full, k, v = _rand((1, 1, nk, 4), 14), _rand((1, 1, nk, 4), 15), _rand((1, 1, nk, 4), 16)
    do = _rand((1, 1, nq, 4), 17)
    do_full = np.zeros((1, 1, nk, 4))
    do_full[:, :, q_start:] = do
    dq, dk, dv = attention_dense_backward(q_full[:, :, q_start:], k, v, do, causal=True, q_start=q_start)
    dq_f, dk_f, dv_f = attention_dense_backward(q_full, k, v, do_full, causal=True)
    assert np.abs(dq - dq_f[:, :, q_start:]).max() < 1e-13
    assert np.abs(dk - dk_f).max() < 1e-13
    assert np.abs(dv - dv_f).max() < 1e-13
