"""bench.py's CPU legs: --oracle-configs (the oracle's per-workload wall-clock report) and the
reference arm's JSON line.

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


def test_reference_arm_line_follows_the_contract(monkeypatch, capsys):
    """bench.py --impl reference times the oracle and prints one JSON line with the
    contract's keys. The line has impl = reference, the GPU arm's metric, unit and
    direction, a cpu_baseline describing the run, and an e2e object with zero copy
    bytes. Tiny stand-ins of the bench's two workloads keep it fast."""
    import bench
    from exact_attention_flash_gb300 import workloads as wl

    tiny = dict(wl.WORKLOADS)
    tiny[bench.FWD_BWD] = wl.Workload(bench.FWD_BWD, "attention", 1, 2, 96, 64, seed=2, causal=True, backward=True,
                                      qk_mult=8.0)
    tiny[bench.DECODE] = wl.Workload(bench.DECODE, "decode", 1, 8, 300, 64, seed=4, n_split=4)
    monkeypatch.setattr(wl, "WORKLOADS", tiny)
    args = type("A", (), {"steps": 2, "warmup": 1, "impl": "reference"})()
    bench.run_reference(args, 1, 0)
    lines = [json.loads(x) for x in capsys.readouterr().out.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    r = lines[0]
    assert r["impl"] == "reference" and r["metric"] == bench.METRIC and r["unit"] == "TFLOP/s"
    assert r["higher_is_better"] is True and r["steps"] == 2 and r["warmup"] == 1 and r["n_gpus"] == 1
    assert r["value"] > 0 and r["dtype"] == "f64" and r["config"]["workload"] == bench.FWD_BWD
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["value"] == r["value"]
    assert r["cpu_baseline"]["cores"] >= 1 and r["cpu_baseline"]["sample"]
    assert r["e2e"] == {"value": r["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_parity_leg_reports_errors_against_the_bars():
    """The bench's oracle leg on tiny samples: outputs equal to the oracle's are within
    the bars; a perturbed O, LSE or gradient is reported over them."""
    import numpy as np

    import bench
    from oracle import attention_dense, attention_dense_backward, attention_split_decode

    rng = np.random.default_rng(0)
    q, k, v, do = (rng.standard_normal((40, 64)) for _ in range(4))
    o, lse = attention_dense(q, k, v, causal=True)
    grads = attention_dense_backward(q, k, v, do, causal=True)
    qd, kd, vd = rng.standard_normal((3, 1, 64)), rng.standard_normal((3, 50, 64)), rng.standard_normal((3, 50, 64))
    od, ld, _ = attention_split_decode(qd, kd, vd, 4)

    def samples(do_shift=0.0, lse_shift=0.0, dk_scale=1.0):
        return {
            "fb": {"kind": "attention", "causal": True, "o_dtype": "bf16", "subset": "tiny",
                   "inputs": {"q": q, "k": k, "v": v, "do": do},
                   "gpu": {"o": o + do_shift, "lse": lse + lse_shift, "dq": grads[0], "dk": grads[1] * dk_scale,
                           "dv": grads[2]}},
            "dec": {"kind": "decode", "n_split": 4, "o_dtype": "f32", "subset": "tiny",
                    "inputs": {"q": qd, "k": kd, "v": vd}, "gpu": {"o": od, "lse": ld[..., 0]}},
        }

    # shapes as the bench keeps them: decode O [heads, 1, d], LSE [heads]
    assert od.shape == (3, 1, 64) and ld[..., 0].shape == (3,)
    ok = bench.oracle_parity(samples())
    assert ok["fb"]["within_bars"] and ok["dec"]["within_bars"]
    assert ok["fb"]["o_max_abs"] < 1e-12 and ok["fb"]["dk_rel_fro"] < 1e-12
    assert not bench.oracle_parity(samples(do_shift=0.05))["fb"]["within_bars"]
    assert not bench.oracle_parity(samples(lse_shift=3e-3))["fb"]["within_bars"]
    bad = bench.oracle_parity(samples(dk_scale=1.05))["fb"]
    assert not bad["within_bars"] and abs(bad["dk_rel_fro"] - 0.05) < 1e-9
