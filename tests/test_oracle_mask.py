"""The oracle's causal mask against the textbook one.

A key is hidden when its position exceeds the query's ("attention_kernels.py"
section 2, ``_mask``). For queries at q_start .. q_start + nq - 1 and keys at
k_start .. k_start + nk - 1 that is numpy's strictly-upper-triangular mask
``triu(ones, 1 + q_start - k_start)``: key column j is hidden for row i iff
j > i + q_start - k_start."""
import numpy as np
import pytest

from oracle.attention import causal_mask


@pytest.mark.parametrize("q_start,nq,nk,k_start", [
    (0, 5, 5, 0), (0, 3, 7, 0), (4, 3, 7, 0), (6, 1, 7, 0), (0, 7, 3, 0),
    (10, 4, 6, 8), (3, 5, 4, 5), (0, 1, 1, 0), (100, 2, 3, 0),
])
def test_causal_mask_is_the_shifted_strict_upper_triangle(q_start, nq, nk, k_start):
    expect = np.triu(np.ones((nq, nk), dtype=bool), 1 + q_start - k_start)
    assert np.array_equal(causal_mask(q_start, nq, nk, k_start), expect)


def test_causal_mask_square_case_hides_exactly_the_future():
    m = causal_mask(0, 4, 4)
    assert not m.diagonal().any()              # a query sees its own key
    assert m.sum() == 4 * 3 // 2               # and no key after it
    assert not m[:, 0].any()                   # key 0 is visible to every query
