"""The oracle's blocked online softmax ("attention_kernels.py" section 3
``flash_forward``: running max, rescale of the accumulated output and sum by
exp(m_old - m_new)) against the dense definition on the score ladders of the GPU
rescale test: whole key tiles at one score, with running-max jumps of about 95 and
140 log2 units.  On the "comparable" ladders the earlier tiles still hold about a
fifth of the weight when the max jumps, so an online softmax that dropped or
mis-scaled what it had accumulated would miss O by about 0.8."""
import numpy as np
import pytest

from oracle import attention_dense, attention_flash_blocked
from tests.test_gpu_rescale import LADDERS, inputs_cpu


@pytest.mark.parametrize("kind,d", sorted(LADDERS))
@pytest.mark.parametrize("bc", [64, 128])
def test_blocked_matches_dense_on_rescale_ladders(kind, d, bc):
    q, k, v = (t.double().numpy()[0, 0] for t in inputs_cpu(kind, d))  # one head: [N, d]
    ref_o, ref_l = attention_dense(q, k, v)
    o, lse = attention_flash_blocked(q, k, v, 128, bc)
    assert np.max(np.abs(o - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12 * np.max(np.abs(ref_l))


def test_comparable_ladder_is_sensitive_to_dropping_earlier_tiles():
    """The pin above has teeth: leaving out the tiles before the jump moves O by far
    more than any tolerance in use."""
    q, k, v = (t.double().numpy() for t in inputs_cpu("comparable", 64))
    ref_o, _ = attention_dense(q, k, v)
    last_o, _ = attention_dense(q, k[:, :, 256:], v[:, :, 256:])
    assert np.max(np.abs(ref_o - last_o)) > 0.5
