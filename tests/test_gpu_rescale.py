"""The forward's held-back reference max and its rescales of O, against the dense
oracle at the usual bars.

The kernel moves a row's reference max only when a key tile's max passes it by more
than 2^32, and then sets it 2^64 above that tile's max; O is rescaled by
2^(m_old - m_new), which flushes to zero on jumps above 2^62.  These inputs put every
key of a 128-key tile at one score, so each row's running max follows a chosen
ladder (in log2 units, score * scale * log2(e)):

- "comparable": tiles at 0, about 95 and about 97.  The second tile stays under the
  reference (0 + 64) + 32 = 96, the third passes it, and the second tile's terms are
  then about 2^-2 of the third's: a rescale that dropped or mis-scaled the terms
  already in O would move O by a large fraction of a V row.
- "flush": tiles at 0, 0 and about 140.  The rescale factor 2^(64 - 204) flushes to
  zero, and the terms it drops are 2^-140 of the new ones.

V rows carry a different offset per key tile, so O tells the tiles' weights apart.
"""
import numpy as np
import pytest
import torch

from oracle import attention_dense
from tests.gpu_util import LSE_MAX_ABS, O_MAX_ABS, f64, max_abs, require_gpu

pytestmark = pytest.mark.gpu

# K[..., 0] per key tile (bf16-exact); Q[..., 0] = 32 for every row, the other
# features of Q are 0, so a key's score is 32 * K[key, 0].
LADDERS = {
    ("comparable", 64): (0.0, 16.5, 16.875),      # log2 units 0, 95.2, 97.4 (scale 1/8)
    ("comparable", 128): (0.0, 23.25, 23.75),     # 0, 94.9, 96.9 (scale 1/sqrt(128))
    ("flush", 64): (0.0, 0.0, 24.25),             # 0, 0, 139.9
    ("flush", 128): (0.0, 0.0, 34.25),            # 0, 0, 139.8
}
V_OFFSET = (0.0, 2.0, -2.0)  # added to every V row of key tile t


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def inputs_cpu(kind, d, rows=256, seed=7):
    """q [1, 1, rows, d], k and v [1, 1, 128 * tiles, d], bf16 on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    ladder = LADDERS[(kind, d)]
    n = 128 * len(ladder)
    q = torch.zeros(1, 1, rows, d)
    q[..., 0] = 32.0
    k = torch.randn(1, 1, n, d, generator=g)
    k[..., 0] = torch.tensor(ladder).repeat_interleave(128)
    v = torch.randn(1, 1, n, d, generator=g) + torch.tensor(V_OFFSET).repeat_interleave(128)[None, None, :, None]
    return tuple(t.to(torch.bfloat16) for t in (q, k, v))


def _inputs(kind, d):
    return tuple(t.cuda() for t in inputs_cpu(kind, d))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", ["comparable", "flush"])
def test_rescale_ladders_match_the_oracle(kind, d):
    from exact_attention_flash_gb300 import fa_device_status, fa_forward

    q, k, v = _inputs(kind, d)
    o, lse = fa_forward(q, k, v, causal=False, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert fa_device_status() == 0
    ref_o, ref_l = attention_dense(f64(q), f64(k), f64(v), causal=False)
    assert max_abs(f64(o), ref_o) <= O_MAX_ABS, f"O error {max_abs(f64(o), ref_o):.3e}"
    assert max_abs(f64(lse), ref_l) <= LSE_MAX_ABS
    if kind == "comparable":
        # the second tile holds a fifth of the weight: O sits well away from either
        # tile's V mean, so a dropped or unscaled second tile fails the bar above
        w2 = 1.0 / (1.0 + 2.0 ** (np.log2(np.e) * 32.0 * (LADDERS[(kind, d)][2] - LADDERS[(kind, d)][1]) / np.sqrt(d)))
        assert 0.1 < w2 < 0.3
