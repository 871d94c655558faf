"""bench.py --oracle-configs on CPU: the oracle's per-workload wall-clock report.

Tiny stand-ins for the named workloads keep this fast. The test checks:
- one JSON line per workload;
- the forms timed for each kind;
- the extrapolation of the row-wise sample: R query rows of a head stand for it
  with a factor (N / R)^2 under causality and N / R otherwise.
"""
import json
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def test_oracle_configs_report(monkeypatch, capsys):
    import bench
    from exact_attention_flash_gb300 import workloads as wl

    tiny = {w.name: w for w in [
        wl.Workload("fwd_small", "attention", 1, 2, 96, 64, seed=0, out_f32=True),
        wl.Workload("causal_fwdbwd_small", "attention", 2, 1, 80, 64, seed=1, causal=True, backward=True),
        wl.Workload("decode_small", "decode", 1, 8, 300, 64, seed=4, n_split=4),
    ]}
    monkeypatch.setattr(wl, "WORKLOADS", tiny)
    bench.run_oracle_configs()
    lines = [json.loads(x) for x in capsys.readouterr().out.splitlines() if x.startswith("{")]
    assert [r["oracle_timing"] for r in lines] == list(tiny)
    for r in lines:
        assert r["kind"] == "oracle" and r["cores"] >= 1
    fwd, fb, dec = lines
    assert fwd["pass"] == "forward" and fb["pass"] == "forward+backward"
    for r in (fwd, fb):
        for k in ("dense_s", "blocked_s", "rowwise_s"):
            assert r[k] > 0
    # N = 96 and 80 are below the row-wise sample sizes: whole heads, factor 1
    assert "the first 96 query rows" in fwd["sample"] and "the first 80 query rows" in fb["sample"]
    assert dec["split_decode_s"] > 0 and dec["dense_s"] > 0 and "8 of 8 heads" in dec["sample"]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [100, 2048, 8192, 16384])
def test_rowwise_extrapolation_matches_pair_counts(causal, N):
    """The factor against the exact count of (query, key) pairs visited: the first R
    rows against all N rows of a head."""
    import bench

    rows, factor = bench.rowwise_sample(N, causal)
    assert 1 <= rows <= N
    if causal:
        exact = (N * (N + 1) / 2) / (rows * (rows + 1) / 2)
    else:
        exact = (N * N) / (rows * N)
    assert abs(factor / exact - 1.0) <= 2e-3
