"""Pins for the oracle's forward paths (dense definition and row-wise tiled).

Each test ties the oracle to something other than itself: a value printed on a
page, a closed form derived by hand, a library routine, or an invariance the
pages state.  All CPU, float64.
"""
import math

import numpy as np
import pytest
import scipy.special

from oracle import attention_dense, attention_dense_rows, attention_tiled_rowwise
from tests.golden.fixtures import load

E = math.e


def test_anchor_printed_row0():
    """"flash_attention_numpy.py", receipt 1: row 0 of O prints as [0.910, 0.755] (scale 1)."""
    g = load("anchor_n3_d2.txt")
    dec = int(g["decimals"][0])
    out, _ = attention_dense(g["Q"], g["K"], g["V"], scale=1.0)
    np.testing.assert_array_equal(np.round(out[0], dec), g["O_row0"])
    tiled, _ = attention_tiled_rowwise(g["Q"], g["K"], g["V"], block=2, scale=1.0)
    np.testing.assert_array_equal(np.round(tiled[0], dec), g["O_row0"])


def _anchor_closed_form():
    # Scores (unscaled): row 0 q=(1,0) -> (1, 0, 2); row 1 q=(0,2) -> (2, 2, 0);
    # row 2 q=(1,1) -> (2, 1, 2).  With V rows (1,0), (0,1), (1,1):
    z0 = E + 1 + E**2
    z1 = 2 * E**2 + 1
    z2 = 2 * E**2 + E
    out = np.array(
        [
            [(E + E**2) / z0, (1 + E**2) / z0],
            [(E**2 + 1) / z1, (E**2 + 1) / z1],
            [2 * E**2 / z2, (E + E**2) / z2],
        ]
    )
    lse = np.log([z0, z1, z2])
    return out, lse


def test_anchor_closed_form_full():
    g = load("anchor_n3_d2.txt")
    want_o, want_l = _anchor_closed_form()
    for fn in (lambda: attention_dense(g["Q"], g["K"], g["V"], scale=1.0),
               lambda: attention_tiled_rowwise(g["Q"], g["K"], g["V"], block=2, scale=1.0)):
        out, lse = fn()
        np.testing.assert_allclose(out, want_o, rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse, want_l, rtol=0, atol=1e-14)


def test_anchor_causal_closed_form():
    """Causal anchor: row 0 sees key 0 only (O = V_0, L = S_00 = 1); row 1 sees two
    equal scores 2 (O = mean of V_0, V_1, L = 2 + ln 2); row 2 sees all keys."""
    g = load("anchor_n3_d2.txt")
    full_o, full_l = _anchor_closed_form()
    want_o = np.array([[1.0, 0.0], [0.5, 0.5], full_o[2]])
    want_l = np.array([1.0, 2.0 + math.log(2.0), full_l[2]])
    for block in (1, 2, 3):
        out, lse = attention_tiled_rowwise(g["Q"], g["K"], g["V"], block=block, scale=1.0, causal=True)
        np.testing.assert_allclose(out, want_o, atol=1e-14)
        np.testing.assert_allclose(lse, want_l, atol=1e-14)
    out, lse = attention_dense(g["Q"], g["K"], g["V"], scale=1.0, causal=True)
    np.testing.assert_allclose(out, want_o, atol=1e-14)
    np.testing.assert_allclose(lse, want_l, atol=1e-14)


def test_uniform_scores_give_mean_of_v():
    """"lab.py" main(): equal scores give the mean of V (= 4 for V = 1, 4, 7)."""
    g = load("uniform_scores.txt")
    out, lse = attention_dense(g["Q"], g["K"], g["V"])
    np.testing.assert_allclose(out, g["O"], atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(3.0)], atol=1e-15)
    for block in (1, 2, 3, 4):
        out, _ = attention_tiled_rowwise(g["Q"], g["K"], g["V"], block=block)
        np.testing.assert_allclose(out, g["O"], atol=1e-15)


def test_single_key_returns_value_and_score():
    rng = np.random.default_rng(11)
    q, k, v = rng.normal(size=(1, 5)), rng.normal(size=(1, 5)), rng.normal(size=(1, 3))
    scale = 0.37
    for out, lse in (attention_dense(q, k, v, scale=scale), attention_tiled_rowwise(q, k, v, 1, scale=scale)):
        np.testing.assert_allclose(out, v, atol=1e-15)
        np.testing.assert_allclose(lse, [scale * float(q[0] @ k[0])], atol=1e-15)


def test_first_causal_row_is_first_value():
    rng = np.random.default_rng(12)
    q, k, v = (rng.normal(size=(9, 4)) for _ in range(3))
    out, lse = attention_dense(q, k, v, causal=True)
    np.testing.assert_allclose(out[0], v[0], atol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * float(q[0] @ k[0]), atol=1e-15)


def _scores_by_loops(q, k, scale, causal):
    n, m = q.shape[0], k.shape[0]
    s = np.empty((n, m))
    for i in range(n):
        for j in range(m):
            s[i, j] = -np.inf if (causal and j > i) else scale * sum(q[i, t] * k[j, t] for t in range(q.shape[1]))
    return s


@pytest.mark.parametrize("causal", [False, True])
def test_dense_matches_scipy_softmax_and_logsumexp(causal):
    rng = np.random.default_rng(13)
    q, k, v = (rng.normal(size=(2, 3, 17, 8)) for _ in range(3))
    out, lse = attention_dense(q, k, v, causal=causal)
    for b in range(2):
        for h in range(3):
            s = _scores_by_loops(q[b, h], k[b, h], 1 / math.sqrt(8), causal)
            np.testing.assert_allclose(lse[b, h], scipy.special.logsumexp(s, axis=1), atol=1e-13)
            np.testing.assert_allclose(out[b, h], scipy.special.softmax(s, axis=1) @ v[b, h], atol=1e-13)


def test_dense_rows_match_dense():
    rng = np.random.default_rng(14)
    q, k, v = (rng.normal(size=(40, 8)) for _ in range(3))
    rows = [0, 1, 17, 39]
    for causal in (False, True):
        full_o, full_l = attention_dense(q, k, v, causal=causal)
        o, l = attention_dense_rows(q, k, v, rows, causal=causal)
        np.testing.assert_allclose(o, full_o[rows], atol=1e-14)
        np.testing.assert_allclose(l, full_l[rows], atol=1e-14)


@pytest.mark.parametrize("n", [5, 6, 7, 33])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_is_block_size_invariant(n, causal):
    """"model.py" verify() and "lab.py": the tiled result equals the dense one at 1e-12
    for blocks 1, 2, 3, 4, 8 (and blocks with an uneven last tile or larger than N)."""
    rng = np.random.default_rng(100 + n)
    q, k, v = (rng.normal(size=(n, 4)) for _ in range(3))
    ref_o, ref_l = attention_dense(q, k, v, causal=causal)
    for block in (1, 2, 3, 4, 5, 8, 16, 64):
        out, lse = attention_tiled_rowwise(q, k, v, block, causal=causal)
        np.testing.assert_allclose(out, ref_o, atol=1e-12, rtol=1e-12)
        np.testing.assert_allclose(lse, ref_l, atol=1e-12, rtol=1e-12)


def test_large_logits_stay_finite_and_exact():
    """"model.py" verify(): q, k x100 stays finite and matches dense at 1e-10."""
    rng = np.random.default_rng(4)
    for n in (5, 6):
        q, k, v = (rng.normal(size=(n, 4)) for _ in range(3))
        ref, ref_l = attention_dense(q * 100, k * 100, v)
        assert np.isfinite(ref).all() and np.isfinite(ref_l).all()
        for causal in (False, True):
            ref, _ = attention_dense(q * 100, k * 100, v, causal=causal)
            out, lse = attention_tiled_rowwise(q * 100, k * 100, v, 2, causal=causal)
            assert np.isfinite(out).all() and np.isfinite(lse).all()
            np.testing.assert_allclose(out, ref, atol=1e-10, rtol=1e-10)


def test_fire_test_big_scores():
    """"flash_attention_numpy.py" receipt 2: Q ~ N(100, 1), K ~ N(0, 1)/8, (64, 8),
    unscaled, tiles of 16: tiled equals dense at 1e-10."""
    rng = np.random.default_rng(0)
    q = rng.normal(100, 1, (64, 8))
    k = rng.normal(0, 1, (64, 8)) / 8
    v = rng.normal(0, 1, (64, 8))
    ref, _ = attention_dense(q, k, v, scale=1.0)
    out, _ = attention_tiled_rowwise(q, k, v, 16, scale=1.0)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, atol=1e-10)


def test_key_shift_invariance():
    """Adding one vector c to every key leaves O unchanged and shifts L_i by scale * q_i . c."""
    rng = np.random.default_rng(15)
    q, k, v = (rng.normal(size=(2, 11, 6)) for _ in range(3))
    c = rng.normal(size=6)
    for causal in (False, True):
        o1, l1 = attention_dense(q, k, v, causal=causal)
        o2, l2 = attention_dense(q, k + c, v, causal=causal)
        np.testing.assert_allclose(o2, o1, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, (q @ c) / math.sqrt(6), atol=1e-12)


def test_rejects_bad_block():
    with pytest.raises(ValueError):
        attention_tiled_rowwise(np.zeros((2, 2)), np.zeros((2, 2)), np.zeros((2, 2)), 0)
