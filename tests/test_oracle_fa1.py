"""Pins of the oracle's key-major loop ("flash_attention_numpy.py"
``flash_attention_tier1``, the first algorithm's order; scale and causal mask as
in "attention_kernels.py" section 3): the page's printed worked example with
tiles of 2, and equality with the dense definition for even and uneven blocks
with and without the causal mask."""
import numpy as np
import pytest

from oracle import attention_dense, attention_fa1_keymajor
from tests.golden.fixtures import load


def test_worked_example_tiles_of_two():
    g = load("anchor_n3_d2.txt")
    o, lse = attention_fa1_keymajor(g["Q"], g["K"], g["V"], 2, 2, scale=1.0)
    assert np.array_equal(np.round(o[0], int(g["decimals"][0])), g["O_row0"])
    # and the rest of the example, as the dense definition gives it
    od, ld = attention_dense(g["Q"], g["K"], g["V"], scale=1.0)
    assert np.abs(o - od).max() < 1e-14 and np.abs(lse - ld).max() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("br,bc", [(1, 1), (2, 3), (4, 4), (5, 7), (8, 2), (64, 128)])
def test_keymajor_equals_dense(br, bc, causal):
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((37, 8)) for _ in range(3))
    o, lse = attention_fa1_keymajor(q, k, v, br, bc, causal=causal)
    od, ld = attention_dense(q[None, None], k[None, None], v[None, None], causal=causal)
    assert np.abs(o - od[0, 0]).max() < 1e-12
    assert np.abs(lse - ld[0, 0]).max() < 1e-12


def test_large_logits_stay_finite():
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((20, 4)) for _ in range(3))
    o, lse = attention_fa1_keymajor(100 * q, k, v, 3, 4, causal=True)
    od, ld = attention_dense(100 * q[None, None], k[None, None], v[None, None], causal=True)
    assert np.isfinite(o).all() and np.abs(o - od[0, 0]).max() < 1e-10
