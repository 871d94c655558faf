"""Pins for the oracle's softmax-state algebra and split-KV decoding.

"attention_kernels.py" section 1 states that merge_states is associative and
commutative with the empty state (-inf, 0, 0) as identity; section 5 splits the
keys at round(Nk * s / n_split) and folds the segment states left to right.
"""
import numpy as np
import pytest

from oracle import (
    SoftmaxState,
    attention_dense,
    attention_split_decode,
    empty_state,
    merge_states,
    split_bounds,
    state_of_scores,
)


def _random_state(rng, shape, dv, empty_mask=None):
    m = rng.normal(scale=5.0, size=shape)
    l = rng.uniform(0.5, 3.0, size=shape)
    o = rng.normal(size=shape + (dv,))
    if empty_mask is not None:
        m = np.where(empty_mask, -np.inf, m)
        l = np.where(empty_mask, 0.0, l)
        o = np.where(empty_mask[..., None], 0.0, o)
    return SoftmaxState(m, l, o)


def _close(a: SoftmaxState, b: SoftmaxState, tol=1e-12):
    np.testing.assert_array_equal(a.m, b.m)
    np.testing.assert_allclose(a.l, b.l, rtol=tol, atol=tol)
    np.testing.assert_allclose(a.o, b.o, rtol=tol, atol=tol)


def test_merge_identity_commutativity_associativity():
    rng = np.random.default_rng(5)
    shape, dv = (4, 6), 5
    empty = rng.uniform(size=shape) < 0.25
    a = _random_state(rng, shape, dv, empty)
    b = _random_state(rng, shape, dv, np.roll(empty, 1))
    c = _random_state(rng, shape, dv)
    e = empty_state(shape, dv)
    _close(merge_states(a, e), a, 0)
    _close(merge_states(e, a), a, 0)
    _close(merge_states(e, e), e, 0)
    _close(merge_states(a, b), merge_states(b, a))
    _close(merge_states(merge_states(a, b), c), merge_states(a, merge_states(b, c)))


def test_state_of_scores_definition():
    """State of a run by its definition; merging two runs' states equals the state
    of their concatenation (the property split decoding relies on)."""
    rng = np.random.default_rng(6)
    s = rng.normal(scale=3.0, size=(3, 10))
    v = rng.normal(size=(10, 4))
    st = state_of_scores(s, v)
    m = s.max(axis=1)
    np.testing.assert_array_equal(st.m, m)
    np.testing.assert_allclose(st.l, np.exp(s - m[:, None]).sum(axis=1), rtol=1e-15)
    np.testing.assert_allclose(st.o, np.exp(s - m[:, None]) @ v, rtol=1e-14)
    left, right = state_of_scores(s[:, :4], v[:4]), state_of_scores(s[:, 4:], v[4:])
    _close(merge_states(left, right), st)


def test_split_bounds_follow_python_round():
    assert split_bounds(10, 4) == [0, 2, 5, 8, 10]  # 2.5 -> 2 and 7.5 -> 8 (half to even)
    assert split_bounds(32768, 64) == list(range(0, 32769, 512))
    for nk in range(0, 40):
        for n_split in range(1, 12):
            assert split_bounds(nk, n_split) == [round(nk * s / n_split) for s in range(n_split + 1)]
    with pytest.raises(ValueError):
        split_bounds(8, 0)


@pytest.mark.parametrize("n_split", [1, 2, 3, 7, 64, 45])
def test_split_decode_equals_dense(n_split):
    rng = np.random.default_rng(9)
    q = rng.normal(size=(2, 3, 1, 16))
    k = rng.normal(size=(2, 3, 40, 16))
    v = rng.normal(size=(2, 3, 40, 16))
    ref_o, ref_l = attention_dense(q, k, v)
    out, lse, parts = attention_split_decode(q, k, v, n_split)
    np.testing.assert_allclose(out, ref_o, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, atol=1e-13)
    bounds = split_bounds(40, n_split)
    for s, part in enumerate(parts):
        j0, j1 = bounds[s], bounds[s + 1]
        if j1 == j0:
            assert np.all(np.isneginf(part.m)) and np.all(part.l == 0) and np.all(part.o == 0)
            continue
        seg_o, seg_l = attention_dense(q, k[..., j0:j1, :], v[..., j0:j1, :])
        np.testing.assert_allclose(part.o / part.l[..., None], seg_o, atol=1e-13)
        np.testing.assert_allclose(part.m + np.log(part.l), seg_l, atol=1e-13)


def test_split_decode_large_logits():
    rng = np.random.default_rng(10)
    q = rng.normal(size=(1, 1, 1, 8)) * 30
    k = rng.normal(size=(1, 1, 50, 8)) * 30
    v = rng.normal(size=(1, 1, 50, 8))
    ref_o, ref_l = attention_dense(q, k, v)
    out, lse, _ = attention_split_decode(q, k, v, 6)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref_o, atol=1e-12)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-14)


def test_split_decode_rejects_bad_split():
    with pytest.raises(ValueError):
        attention_split_decode(np.zeros((1, 4)), np.zeros((3, 4)), np.zeros((3, 4)), 0)
