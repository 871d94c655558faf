#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = the whole path once: causal forward and backward on the
B=2, H=16, N=8192, d=128 workload (Q and K x8, seed 2) and split-KV decode on
the B=16, H=32, L=32768, d=128, 64-split workload (seed 4).  The headline value
is forward+backward TFLOP/s (FLOPs 4*B*H*N^2*d, halved when causal, x2.5 for
the backward); decode is reported as HBM GB/s in its own sub-object.

Prints one JSON line (rank 0).  `--impl reference` times the float64 CPU
oracle instead (bounded sample of the same workload, host cores).
Under torchrun each rank runs an independent replica (the path needs no
exchange between GPUs); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

_NCORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_NCORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_NCORES))

import torch  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s & % of bf16 TC peak; decode HBM GB/s"
FWD_BWD = "causal_fwdbwd_b2h16_n8192_d128_qk8"
DECODE = "decode_b16h32_l32768_d128_s64"


def attention_flops(B, H, N, d, causal, backward):
    """Matmul FLOPs of attention: 4*N^2*d per head forward, 2.5x that backward
    (recompute included), halved when causal; softmax exps not counted."""
    f = 4.0 * B * H * N * N * d
    if backward:
        f *= 2.5
    return f / 2 if causal else f


def decode_bytes(B, H, L, d, n_split):
    """Algorithmic HBM bytes of one decode: K and V read once (bf16), q read,
    O (fp32) and LSE written, segment states written and read back."""
    kv = 2 * B * H * L * d * 2
    q = B * H * d * 2
    out = B * H * d * 4 + B * H * 4
    states = 2 * B * H * n_split * (d + 2) * 4
    return kv + q + out + states


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        j = json.loads(p.read_text())
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_sha(name):
    return hashlib.sha256((ROOT / "exact_attention_flash_gb300" / "csrc" / name).read_bytes()).hexdigest()[:16]


def recorded_traffic(kernel_file, key):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel source is unchanged since."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    rec = json.loads(p.read_text()).get(key)
    if not rec or rec.get("source_sha") != source_sha(kernel_file):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- bars of the path
O_MAX_ABS, LSE_MAX_ABS, GRAD_REL_FRO = 1e-2, 2e-3, 2e-2


def _bf16_half_ulp(x):
    """Half a bf16 ulp at |x| (8 significant bits): the storage rounding of a bf16 output."""
    import numpy as np

    x = np.abs(np.asarray(x, dtype=np.float64))
    return 2.0 ** (np.floor(np.log2(np.maximum(x, 2.0 ** -126))) - 8)


def _rel_fro(got, ref):
    import numpy as np

    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def oracle_parity(samples):
    """The cpu_baseline leg: the float64 oracle on each workload's sample (heads of the
    very inputs the GPU ran, with the GPU's outputs for them), timed, and the GPU's
    errors against it at the path's bars (O max-abs 1e-2, plus bf16's half-ulp for a
    bf16 output; LSE max-abs 2e-3; dQ, dK, dV relative Frobenius 2e-2)."""
    import numpy as np

    from oracle import attention_dense, attention_dense_backward, attention_split_decode

    out = {}
    for name, smp in samples.items():
        x, g = smp["inputs"], smp["gpu"]
        t0 = time.perf_counter()
        if smp["kind"] == "decode":
            ref_o, ref_l, _ = attention_split_decode(x["q"], x["k"], x["v"], smp["n_split"])
            ref_l = ref_l[..., 0]
            grads = None
        else:
            ref_o, ref_l = attention_dense(x["q"], x["k"], x["v"], causal=smp["causal"])
            grads = (attention_dense_backward(x["q"], x["k"], x["v"], x["do"], causal=smp["causal"])
                     if "do" in x else None)
        secs = time.perf_counter() - t0
        err_o = np.abs(g["o"] - ref_o)
        bar = O_MAX_ABS + (_bf16_half_ulp(ref_o) if smp["o_dtype"] == "bf16" else 0.0)
        par = {"subset": smp["subset"], "o_dtype": smp["o_dtype"], "o_max_abs": float(err_o.max()),
               "o_excess_over_bar": float((err_o - bar).max()), "lse_max_abs": float(np.abs(g["lse"] - ref_l).max())}
        ok = par["o_excess_over_bar"] <= 0 and par["lse_max_abs"] <= LSE_MAX_ABS
        if grads is not None:
            for gname, ref in zip(("dq", "dk", "dv"), grads):
                par[gname + "_rel_fro"] = _rel_fro(g[gname], ref)
                ok = ok and par[gname + "_rel_fro"] <= GRAD_REL_FRO
        par["within_bars"] = bool(ok)
        par["oracle_seconds"] = secs
        out[name] = par
    return out


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(w_fb, w_dec, n_heads_fb, n_heads_dec):
    """Run the float64 oracle on `n_heads` heads of each workload; return
    (seconds, algorithmic fwd+bwd FLOPs of the sample, decode bytes of the sample)."""
    import numpy as np

    from exact_attention_flash_gb300.workloads import make_attention_inputs, make_decode_inputs
    from oracle import attention_dense, attention_dense_backward, attention_split_decode

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v, do = make_attention_inputs(1, n_heads_fb, w_fb.N, w_fb.d, w_fb.seed, dev, qk_mult=w_fb.qk_mult)
    q, k, v, do = (t.double().cpu().numpy() for t in (q, k, v, do))
    qd, kd, vd = make_decode_inputs(1, n_heads_dec, w_dec.N, w_dec.d, w_dec.seed, dev)
    qd, kd, vd = (t.double().cpu().numpy() for t in (qd, kd, vd))
    t0 = time.perf_counter()
    attention_dense(q, k, v, causal=True)
    attention_dense_backward(q, k, v, do, causal=True)
    t1 = time.perf_counter()
    attention_split_decode(qd, kd, vd, w_dec.n_split)
    t2 = time.perf_counter()
    flops = attention_flops(1, n_heads_fb, w_fb.N, w_fb.d, True, False) + attention_flops(
        1, n_heads_fb, w_fb.N, w_fb.d, True, True)
    dbytes = decode_bytes(1, n_heads_dec, w_dec.N, w_dec.d, w_dec.n_split)
    del np
    return t1 - t0, t2 - t1, flops, dbytes


def cpu_baseline_record(heads_fb=1, heads_dec=8):
    from exact_attention_flash_gb300.workloads import WORKLOADS

    w_fb, w_dec = WORKLOADS[FWD_BWD], WORKLOADS[DECODE]
    t_fb, t_dec, flops, dbytes = oracle_sample(w_fb, w_dec, heads_fb, heads_dec)
    return {
        "value": flops / t_fb / 1e12,
        "unit": "TFLOP/s",
        "cores": _NCORES,
        "kind": "oracle",
        "sample": f"{heads_fb} of {w_fb.B * w_fb.H} heads of {FWD_BWD} (forward+backward, float64 numpy, "
                  f"{t_fb:.2f} s); decode: {heads_dec} of {w_dec.B * w_dec.H} heads of {DECODE} ({t_dec:.2f} s, "
                  f"{dbytes / t_dec / 1e9:.3f} GB/s)",
        "seconds": t_fb + t_dec,
        "decode_gbs": dbytes / t_dec / 1e9,
    }


def rowwise_sample(n, causal):
    """Query rows of one head that the row-wise oracle is timed on, and the factor from
    their time to the head's: under causality row i visits i + 1 keys, so the first R
    rows do about (R / N)^2 of the head's work; otherwise every row visits N keys."""
    rows = min(n, 1024 if causal else 256)
    return rows, ((n / rows) ** 2 if causal else n / rows)


def run_oracle_configs():
    """Wall-clock of the float64 oracle on every named workload, on this host's cores.

    Three oracle forms per workload, each on a bounded sample, extrapolated to the
    whole workload (one JSON line per workload):
    - dense: the definition, whole heads;
    - blocked: the block-tiled online softmax (128 x 128 tiles), whole heads;
    - rowwise: one query row at a time over key tiles of 64. It runs the first R
      query rows of a head. Row i costs in proportion to i + 1 under causality and to
      N otherwise, so the head's time is (N / R)^2 resp. N / R times that.
    Forward and, where the workload has one, backward; decode: the split-KV oracle
    (split and merge) and the dense definition over all keys.
    """
    from exact_attention_flash_gb300.workloads import WORKLOADS, make_attention_inputs, make_decode_inputs
    from oracle import (attention_dense, attention_dense_backward, attention_flash_blocked,
                        attention_flash_blocked_backward, attention_split_decode, attention_tiled_rowwise,
                        attention_tiled_rowwise_backward)

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    for name, w in WORKLOADS.items():
        heads = w.B * w.H
        rec = {"oracle_timing": name, "cores": _NCORES, "kind": "oracle", "dtype": "f64"}
        if w.kind == "decode":
            n_heads = 8
            q, k, v = (t.double().numpy()[0] for t in make_decode_inputs(1, n_heads, w.N, w.d, w.seed, "cpu"))
            t_split = timed(lambda: attention_split_decode(q[None], k[None], v[None], w.n_split))
            t_dense = timed(lambda: attention_dense(q, k, v))
            work = decode_bytes(1, n_heads, w.N, w.d, w.n_split)
            rec.update({"sample": f"{n_heads} of {heads} heads",
                        "split_decode_s": t_split * heads / n_heads, "dense_s": t_dense * heads / n_heads,
                        "split_decode_gbs": work / t_split / 1e9})
        else:
            q, k, v, do = (t.double().numpy()[0, 0] for t in make_attention_inputs(
                1, 1, w.N, w.d, w.seed, "cpu", qk_mult=w.qk_mult))
            c = w.causal
            rows, grow = rowwise_sample(w.N, c)
            t_dense = timed(lambda: attention_dense(q, k, v, causal=c))
            t_block = timed(lambda: attention_flash_blocked(q, k, v, 128, 128, causal=c))
            o_r, l_r = attention_tiled_rowwise(q[:rows], k, v, 64, causal=c)
            t_row = timed(lambda: attention_tiled_rowwise(q[:rows], k, v, 64, causal=c))
            flops = attention_flops(1, 1, w.N, w.d, c, False)
            if w.backward:
                o, lse = attention_dense(q, k, v, causal=c)
                t_dense += timed(lambda: attention_dense_backward(q, k, v, do, causal=c))
                t_block += timed(lambda: attention_flash_blocked_backward(q, k, v, o, lse, do, 128, 128, causal=c))
                t_row += timed(lambda: attention_tiled_rowwise_backward(q[:rows], k, v, o[:rows], lse[:rows],
                                                                        do[:rows], 64, causal=c))
                flops += attention_flops(1, 1, w.N, w.d, c, True)
            del o_r, l_r
            rec.update({"sample": f"1 of {heads} heads; rowwise: the first {rows} query rows of it",
                        "pass": "forward+backward" if w.backward else "forward",
                        "dense_s": t_dense * heads, "blocked_s": t_block * heads, "rowwise_s": t_row * grow * heads,
                        "dense_tflops": flops / t_dense / 1e12, "blocked_tflops": flops / t_block / 1e12,
                        "rowwise_tflops": flops / (t_row * grow) / 1e12})
        print(json.dumps(rec), flush=True)


def run_reference(args, world, rank):
    if rank != 0:
        return
    from exact_attention_flash_gb300.workloads import WORKLOADS

    w_fb = WORKLOADS[FWD_BWD]
    for _ in range(args.warmup):
        cpu_baseline_record(heads_fb=1, heads_dec=4)
    vals, secs = [], []
    rec = None
    for _ in range(args.steps):
        rec = cpu_baseline_record(heads_fb=1, heads_dec=4)
        vals.append(rec["value"])
        secs.append(rec["seconds"])
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.median(secs),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded, widened to float64)",
        "config": {"workload": FWD_BWD, "B": w_fb.B, "H": w_fb.H, "N": w_fb.N, "d": w_fb.d, "causal": True,
                   "decode_workload": DECODE, "sample": rec["sample"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": rec["cores"], "kind": "oracle",
                         "sample": rec["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU path
def _time_alone(fn, reps, flush, stream):
    """Median and best of `reps` CUDA-event timings of fn() on `stream`, after 3
    warm-up calls, with L2 flushed (a 256 MB write) before each timed call."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        fn()
    times = []
    for _ in range(reps):
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times), min(times)


def _rate_record(med_ms, best_ms, work, unit, peaks, reps):
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    r = {"median_ms": med_ms, "best_ms": best_ms, "reps": reps, "unit": unit, "rate": work / (med_ms * 1e-3) / scale,
         "best_rate": work / (best_ms * 1e-3) / scale}
    if unit == "TFLOP/s":
        r["frac_of_bf16_peak"] = r["rate"] / peaks["bf16_tflops"]
        r["frac_of_bf16_sustained"] = r["rate"] / peaks["bf16_tflops_sustained"]
    else:
        r["frac_of_hbm_peak"] = r["rate"] / peaks["hbm_gbs"]
        r["frac_of_8tbs"] = r["rate"] / 8000.0
    return r


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def workload_records(peaks, reps, dev, stream, keep_samples):
    """Every named workload's kernels, each timed alone (median and best of `reps`,
    L2 flushed before each call), with the GPU's outputs for a few heads kept (as
    float64 host arrays, inputs alongside) for the oracle leg's parity check."""
    from exact_attention_flash_gb300 import (backward_workspace_bytes, decode_workspace_bytes, fa_backward,
                                             fa_decode, fa_forward, forward_workspace_bytes)
    from exact_attention_flash_gb300.workloads import WORKLOADS, make_inputs

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    recs, samples = {}, {}
    for name, w in WORKLOADS.items():
        if w.kind == "decode":
            q, k, v = make_inputs(w, dev)
            ws = torch.empty(decode_workspace_bytes(w.B, w.H, w.d, w.n_split), device=dev, dtype=torch.uint8)
            o = torch.empty((w.B, w.H, 1, w.d), device=dev)
            lse = torch.empty((w.B, w.H), device=dev)
            med, best = _time_alone(lambda: fa_decode(q, k, v, w.n_split, workspace=ws, out=o, lse=lse, stream=stream),
                                    reps, flush, stream)
            recs[name] = {"B": w.B, "H": w.H, "L": w.N, "d": w.d, "n_split": w.n_split, "kernels": {
                "decode": _rate_record(med, best, decode_bytes(w.B, w.H, w.N, w.d, w.n_split), "GB/s", peaks, reps)}}
            heads = [(0, 0), (0, 31), (3, 7), (7, 16), (9, 1), (12, 30), (15, 0), (15, 31)]
            if keep_samples:
                pick = lambda t: _f64(torch.stack([t[b, h] for b, h in heads]))  # noqa: E731
                samples[name] = {"kind": "decode", "n_split": w.n_split, "o_dtype": "f32",
                                 "subset": f"{len(heads)} of {w.B * w.H} heads",
                                 "inputs": {"q": pick(q), "k": pick(k), "v": pick(v)},
                                 "gpu": {"o": pick(o), "lse": _f64(torch.stack([lse[b, h] for b, h in heads]))}}
            del q, k, v, ws, o, lse
        else:
            q, k, v, do = make_inputs(w, dev)
            odt = torch.float32 if w.out_f32 else torch.bfloat16
            o = torch.empty(q.shape, device=dev, dtype=odt)
            lse = torch.empty((w.B, w.H, w.N), device=dev)
            wsf = torch.empty(forward_workspace_bytes(w.B, w.H, w.N, w.d, w.causal), device=dev, dtype=torch.uint8)
            fwd = lambda: fa_forward(q, k, v, causal=w.causal, out=o, lse=lse, workspace=wsf, stream=stream)  # noqa: E731
            med, best = _time_alone(fwd, reps, flush, stream)
            kern = {"forward": _rate_record(med, best, attention_flops(w.B, w.H, w.N, w.d, w.causal, False),
                                            "TFLOP/s", peaks, reps)}
            grads = None
            if w.backward:
                grads = [torch.empty(q.shape, device=dev) for _ in range(3)]
                wsb = torch.empty(backward_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
                bwd = lambda: fa_backward(q, k, v, o, lse, do, causal=w.causal, workspace=wsb,  # noqa: E731
                                          dq=grads[0], dk=grads[1], dv=grads[2], stream=stream)
                med, best = _time_alone(bwd, reps, flush, stream)
                kern["backward"] = _rate_record(med, best, attention_flops(w.B, w.H, w.N, w.d, w.causal, True),
                                                "TFLOP/s", peaks, reps)
            recs[name] = {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal, "qk_mult": w.qk_mult,
                          "o_dtype": "f32" if w.out_f32 else "bf16", "kernels": kern}
            if w.B * w.H == 1:
                recs[name]["note"] = "one (batch, head): two CTAs of 128 rows, launch-latency bound"
            if keep_samples:
                x = {"q": _f64(q[0, 0]), "k": _f64(k[0, 0]), "v": _f64(v[0, 0])}
                g = {"o": _f64(o[0, 0]), "lse": _f64(lse[0, 0])}
                if grads is not None:
                    x["do"] = _f64(do[0, 0])
                    g.update(dq=_f64(grads[0][0, 0]), dk=_f64(grads[1][0, 0]), dv=_f64(grads[2][0, 0]))
                samples[name] = {"kind": "attention", "causal": w.causal, "o_dtype": recs[name]["o_dtype"],
                                 "subset": f"head (0, 0) of {w.B * w.H}", "inputs": x, "gpu": g}
            del q, k, v, do, o, lse, wsf, grads
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return recs, samples


def run_ours(args, world, rank, local):
    from exact_attention_flash_gb300 import (_lib, backward_workspace_bytes, decode_workspace_bytes, fa_backward,
                                             fa_decode, fa_device_status, fa_forward, forward_workspace_bytes)
    from exact_attention_flash_gb300.build import build
    from exact_attention_flash_gb300.workloads import WORKLOADS, make_inputs

    if rank == 0 or world > 1:
        build()
    barrier(world)
    _lib.load()
    dev = torch.device("cuda", local)
    w, wd = WORKLOADS[FWD_BWD], WORKLOADS[DECODE]
    q, k, v, do = make_inputs(w, dev)
    qd, kd, vd = make_inputs(wd, dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    dq = torch.empty(q.shape, device=dev, dtype=torch.float32)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    ws_f = torch.empty(forward_workspace_bytes(w.B, w.H, w.N, w.d, True), device=dev, dtype=torch.uint8)
    ws_b = torch.empty(backward_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
    od = torch.empty((wd.B, wd.H, 1, wd.d), device=dev, dtype=torch.float32)
    lsed = torch.empty((wd.B, wd.H), device=dev, dtype=torch.float32)
    ws_d = torch.empty(decode_workspace_bytes(wd.B, wd.H, wd.d, wd.n_split), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        fa_forward(q, k, v, causal=True, out=o, lse=lse, workspace=ws_f, stream=stream)

    def bwd():
        fa_backward(q, k, v, o, lse, do, causal=True, workspace=ws_b, dq=dq, dk=dk, dv=dv, stream=stream)

    def dec():
        fa_decode(qd, kd, vd, wd.n_split, workspace=ws_d, out=od, lse=lsed, stream=stream)

    for _ in range(max(args.warmup, 3)):
        fwd()
        bwd()
        dec()
    torch.cuda.synchronize(dev)
    if fa_device_status() != 0:
        raise RuntimeError("device status not clean after warm-up")

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(n):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
        dec()
        ev[i][3].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    if fa_device_status() != 0:
        raise RuntimeError("device status not clean after the timed steps")
    t_fwd = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    t_bwd = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    t_dec = [ev[i][2].elapsed_time(ev[i][3]) for i in range(n)]
    t_step = [ev[i][0].elapsed_time(ev[i][3]) for i in range(n)]
    # Medians over the timed steps (best and mean alongside); max over ranks.
    fwd_ms = max_over_ranks(statistics.median(t_fwd), world)
    bwd_ms = max_over_ranks(statistics.median(t_bwd), world)
    dec_ms = max_over_ranks(statistics.median(t_dec), world)
    step_ms = max_over_ranks(statistics.median(t_step), world)

    f_fwd = attention_flops(w.B, w.H, w.N, w.d, True, False)
    f_bwd = attention_flops(w.B, w.H, w.N, w.d, True, True)
    dbytes = decode_bytes(wd.B, wd.H, wd.N, wd.d, wd.n_split)
    value = world * (f_fwd + f_bwd) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    peaks = load_peaks()

    # ---- end to end through the public API with host buffers (pinned), copies timed.
    # Three streams pipeline the steps, as a host feeding the GPU would: step i's
    # inputs are copied in while step i - 1 computes and step i - 2's results are
    # copied out (one copy stream per direction: two streams in the same direction
    # measured slower).  Device inputs and outputs are double-buffered; events order
    # each reuse.  The timed region runs from before the first copy in to after the
    # last copy out, so every step's copies are inside it.
    host_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
    dev_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def make_e2e(grad_dtype):
        """The pipelined end-to-end step for gradients of ``grad_dtype``, and its bytes copied out."""
        ws = ws_b if grad_dtype == torch.float32 else torch.empty(
            backward_workspace_bytes(w.B, w.H, w.N, w.d, grad_dtype), device=dev, dtype=torch.uint8)
        outs = (o, lse) + tuple(torch.empty(t.shape, dtype=grad_dtype, device=dev) for t in (dq, dk, dv))
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _ in range(2)]
        dev_out = [[torch.empty_like(t) for t in outs] for _ in range(2)]

        def run(steps):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            computed = [None, None]  # compute of the last step that read dev_in[b]
            copied = [None, None]    # copy out of the last step that wrote dev_out[b]
            for i in range(steps):
                b = i % 2
                if computed[b] is not None:
                    s_in.wait_event(computed[b])
                with torch.cuda.stream(s_in):
                    for dst, src in zip(dev_in[b], host_in):
                        dst.copy_(src, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
                stream.wait_event(ev_in)
                if copied[b] is not None:
                    stream.wait_event(copied[b])
                x = dev_in[b]
                ob, lb, dqb, dkb, dvb = dev_out[b]
                fa_forward(x[0], x[1], x[2], causal=True, out=ob, lse=lb, workspace=ws_f, stream=stream)
                fa_backward(x[0], x[1], x[2], ob, lb, x[3], causal=True, workspace=ws, dq=dqb, dk=dkb, dv=dvb,
                            stream=stream, grad_dtype=grad_dtype)
                computed[b] = torch.cuda.Event()
                computed[b].record(stream)
                s_out.wait_event(computed[b])
                with torch.cuda.stream(s_out):
                    for dst, src in zip(host_out[b], dev_out[b]):
                        dst.copy_(src, non_blocking=True)
                copied[b] = torch.cuda.Event()
                copied[b].record(s_out)
            done = torch.cuda.Event()
            done.record(s_out)
            stream.wait_event(done)
            end.record(stream)
            return start, end

        return run, sum(t.numel() * t.element_size() for t in host_out[0])

    def e2e_measure(grad_dtype):
        run, d2h = make_e2e(grad_dtype)
        run(2)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = run(n)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1) / n, world)
        return world * (f_fwd + f_bwd) / (ms * 1e-3) / 1e12, d2h

    e2e_value, d2h = e2e_measure(torch.float32)
    e2e16_value, d2h16 = e2e_measure(torch.bfloat16)
    if fa_device_status() != 0:
        raise RuntimeError("device status not clean after the end-to-end steps")

    # ---- every named workload, each kernel timed alone; the oracle leg (cpu_baseline)
    # checks the GPU's outputs on a few heads of each.
    del host_in, dev_in
    torch.cuda.empty_cache()
    want_oracle = rank == 0 and world == 1 and not args.no_cpu_baseline
    per_workload, samples = workload_records(peaks, max(args.reps, 20), dev, stream, keep_samples=want_oracle)
    if fa_device_status() != 0:
        raise RuntimeError("device status not clean after the per-workload timings")

    if rank != 0:
        return
    bwd_tflops = f_bwd / (bwd_ms * 1e-3) / 1e12
    fwd_tflops = f_fwd / (fwd_ms * 1e-3) / 1e12
    dec_gbs = dbytes / (dec_ms * 1e-3) / 1e9
    cpu = None
    if want_oracle:
        parity = oracle_parity(samples)
        for name, par in parity.items():
            per_workload[name]["parity"] = par
        fb, dc = parity[FWD_BWD], parity[DECODE]
        fb_flops = attention_flops(1, 1, w.N, w.d, True, False) + attention_flops(1, 1, w.N, w.d, True, True)
        dc_bytes = decode_bytes(1, 8, wd.N, wd.d, wd.n_split)
        cpu = {"value": fb_flops / fb["oracle_seconds"] / 1e12, "unit": "TFLOP/s", "cores": _NCORES, "kind": "oracle",
               "sample": f"head (0, 0) of {FWD_BWD} (dense forward + backward, float64 numpy, "
                         f"{fb['oracle_seconds']:.2f} s); decode: {dc['subset']} of {DECODE} "
                         f"({dc['oracle_seconds']:.2f} s, {dc_bytes / dc['oracle_seconds'] / 1e9:.3f} GB/s); "
                         "the same runs give each workload's parity errors",
               "seconds": sum(p["oracle_seconds"] for p in parity.values()),
               "decode_gbs": dc_bytes / dc["oracle_seconds"] / 1e9}

    def step_kernel(ts, ms):
        return {"median_ms": ms, "best_ms": min(ts), "mean_ms": sum(ts) / len(ts)}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": n,
        "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16; Q,K x8)",
        "config": {"workload": FWD_BWD, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True,
                   "decode_workload": DECODE, "l2": "inputs larger than L2 (K/V stream of 8.6 GB per step); "
                   "the per-workload timings flush L2 before each call",
                   "timing": "medians over the timed steps", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "fa_backward (preprocess + bwd_kernel)", "achieved": bwd_tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": bwd_tflops / peaks["bf16_tflops"],
                     "traffic": recorded_traffic("fa_bwd.cu", "bwd_kernel_d128_causal"),
                     "peak_source": peaks["source"] + " burst"},
        "kernels": {
            "forward": {**step_kernel(t_fwd, fwd_ms), "ms": fwd_ms, "tflops": fwd_tflops,
                        "frac_of_bf16_peak": fwd_tflops / peaks["bf16_tflops"],
                        "frac_of_bf16_sustained": fwd_tflops / peaks["bf16_tflops_sustained"],
                        "traffic": recorded_traffic("fa_fwd.cu", "fwd_kernel_d128_causal")},
            "backward": {**step_kernel(t_bwd, bwd_ms), "ms": bwd_ms, "tflops": bwd_tflops,
                         "frac_of_bf16_peak": bwd_tflops / peaks["bf16_tflops"],
                         "frac_of_bf16_sustained": bwd_tflops / peaks["bf16_tflops_sustained"]},
            "decode": {**step_kernel(t_dec, dec_ms), "ms": dec_ms, "gbs": dec_gbs, "bound": "hbm",
                       "peak_gbs": peaks["hbm_gbs"], "frac_of_hbm_peak": dec_gbs / peaks["hbm_gbs"],
                       "frac_of_8tbs": dec_gbs / 8000.0, "algorithmic_bytes": dbytes,
                       "traffic": recorded_traffic("fa_decode.cu", "decode_split_kernel_d128")},
        },
        "workloads": per_workload,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "grad_dtype": "f32"},
        # the same pipeline with the gradients returned as bf16 (fp32 accumulation inside)
        "e2e_bf16_grads": {"value": e2e16_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h16},
        # this library's kernels per timed step: fwd_kernel, bwd_preprocess + bwd_kernel,
        # decode_split_kernel (the forward's and the decode's counter clears are runtime memsets)
        "gpu_launches": 4 * n,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# Reduced cases for profiler captures: inputs larger than the 129 MB L2, a few GB on the device.
PROFILE_CASES = {
    "fwd": dict(B=2, H=32, N=4096, d=128, causal=True, qk_mult=8.0, seed=2),
    "fwd_d64": dict(B=4, H=32, N=2048, d=64, causal=True, qk_mult=1.0, seed=1),
    "bwd": dict(B=2, H=32, N=4096, d=128, causal=True, qk_mult=8.0, seed=2),
    "bwd_d64": dict(B=4, H=32, N=2048, d=64, causal=True, qk_mult=1.0, seed=1),
    "decode": dict(B=4, H=32, L=32768, d=128, n_split=64, seed=4),
}


def run_profile_case(name, reps):
    """Launch one kernel family `reps` times on a reduced case (for ncu; prints timing only)."""
    from exact_attention_flash_gb300 import fa_backward, fa_decode, fa_device_status, fa_forward
    from exact_attention_flash_gb300.build import build
    from exact_attention_flash_gb300.workloads import make_attention_inputs, make_decode_inputs

    build()
    c = PROFILE_CASES[name]
    if name == "decode":
        qd, kd, vd = make_decode_inputs(c["B"], c["H"], c["L"], c["d"], c["seed"], "cuda")
        fn = lambda: fa_decode(qd, kd, vd, c["n_split"])  # noqa: E731
    else:
        q, k, v, do = make_attention_inputs(c["B"], c["H"], c["N"], c["d"], c["seed"], "cuda", qk_mult=c["qk_mult"])
        o, lse = fa_forward(q, k, v, causal=c["causal"])
        if name.startswith("fwd"):
            fn = lambda: fa_forward(q, k, v, causal=c["causal"], out=o, lse=lse)  # noqa: E731
        else:
            from exact_attention_flash_gb300 import backward_workspace_bytes

            ws = torch.empty(backward_workspace_bytes(c["B"], c["H"], c["N"], c["d"]), device="cuda", dtype=torch.uint8)
            fn = lambda: fa_backward(q, k, v, o, lse, do, causal=c["causal"], workspace=ws)  # noqa: E731
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if fa_device_status() != 0:
        raise RuntimeError("device status not clean")
    print(json.dumps({"profile_case": name, **c, "reps": reps, "ms_per_call": e0.elapsed_time(e1) / reps}))


def run_all_workloads(reps):
    """One JSON line per named workload and kernel family: each call timed alone
    with CUDA events (median of `reps`), with L2 flushed by a 256 MB write before
    every timed call, so that small workloads are not timed from a warm L2."""
    from exact_attention_flash_gb300 import (backward_workspace_bytes, decode_auto_split, fa_backward, fa_decode,
                                             fa_forward, fa_forward_keymajor, fa_merge_states)
    from exact_attention_flash_gb300.build import build
    from exact_attention_flash_gb300.workloads import WORKLOADS, make_attention_inputs, make_decode_inputs

    build()
    peaks = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Beyond the named workloads: the merge of two fp32 results of the bench forward's
    # shape, and the decode workload with the library's automatic split count.
    extra = {}
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    m_shape = (2, 16, 8192)
    m_in = [torch.randn(m_shape + (128,), generator=g, device="cuda") for _ in range(2)]
    m_lse = [torch.randn(m_shape, generator=g, device="cuda") for _ in range(2)]
    m_out, m_out_lse = torch.empty_like(m_in[0]), torch.empty_like(m_lse[0])
    rows = m_lse[0].numel()
    extra["merge_b2h16_n8192_d128_f32"] = {"merge": (
        lambda: fa_merge_states(m_in[0], m_lse[0], m_in[1], m_lse[1], out=m_out, lse=m_out_lse),  # noqa: E731
        3 * rows * 128 * 4 + 3 * rows * 4, "GB/s")}
    wd = WORKLOADS["decode_b16h32_l32768_d128_s64"]
    qa, ka, va = make_decode_inputs(wd.B, wd.H, wd.N, wd.d, wd.seed, "cuda")
    n_auto = decode_auto_split(wd.B, wd.H, wd.N)
    oa, la = fa_decode(qa, ka, va, n_auto)
    extra[f"decode_b16h32_l32768_d128_auto{n_auto}"] = {"decode": (
        lambda: fa_decode(qa, ka, va, n_auto, out=oa, lse=la),  # noqa: E731
        decode_bytes(wd.B, wd.H, wd.N, wd.d, n_auto), "GB/s")}
    # The first algorithm's key-major loop order on the bench's causal workload, for comparison.
    wk = WORKLOADS["causal_fwdbwd_b2h16_n8192_d128_qk8"]
    qk_, kk_, vk_, _ = make_attention_inputs(wk.B, wk.H, wk.N, wk.d, wk.seed, "cuda", qk_mult=wk.qk_mult,
                                              with_do=False)
    extra["causal_b2h16_n8192_d128_qk8 (key-major order)"] = {"forward_keymajor": (
        lambda: fa_forward_keymajor(qk_, kk_, vk_, causal=True),  # noqa: E731
        attention_flops(wk.B, wk.H, wk.N, wk.d, True, False), "TFLOP/s")}
    for name, w in list(WORKLOADS.items()) + list(extra.items()):
        if isinstance(w, dict):
            calls = w
            _time_calls(name, calls, reps, flush, e0, e1, peaks)
            continue
        calls = {}
        if w.kind == "decode":
            q, k, v = make_decode_inputs(w.B, w.H, w.N, w.d, w.seed, "cuda")
            o, l = fa_decode(q, k, v, w.n_split)
            calls["decode"] = (lambda: fa_decode(q, k, v, w.n_split, out=o, lse=l),  # noqa: E731
                               decode_bytes(w.B, w.H, w.N, w.d, w.n_split), "GB/s")
        else:
            q, k, v, do = make_attention_inputs(w.B, w.H, w.N, w.d, w.seed, "cuda", qk_mult=w.qk_mult,
                                                with_do=w.backward)
            odt = torch.float32 if w.out_f32 else torch.bfloat16
            o, lse = fa_forward(q, k, v, causal=w.causal, out_dtype=odt)
            calls["forward"] = (lambda: fa_forward(q, k, v, causal=w.causal, out=o, lse=lse),  # noqa: E731
                                attention_flops(w.B, w.H, w.N, w.d, w.causal, False), "TFLOP/s")
            if w.backward:
                ws = torch.empty(backward_workspace_bytes(w.B, w.H, w.N, w.d), device="cuda", dtype=torch.uint8)
                calls["backward"] = (lambda: fa_backward(q, k, v, o, lse, do, causal=w.causal, workspace=ws),  # noqa: E731
                                     attention_flops(w.B, w.H, w.N, w.d, w.causal, True), "TFLOP/s")
                ws16 = torch.empty(backward_workspace_bytes(w.B, w.H, w.N, w.d, torch.bfloat16), device="cuda",
                                   dtype=torch.uint8)
                calls["backward (bf16 gradients)"] = (
                    lambda: fa_backward(q, k, v, o, lse, do, causal=w.causal, workspace=ws16,  # noqa: E731
                                        grad_dtype=torch.bfloat16),
                    attention_flops(w.B, w.H, w.N, w.d, w.causal, True), "TFLOP/s")
        _time_calls(name, calls, reps, flush, e0, e1, peaks)
        del calls
        torch.cuda.empty_cache()


def _time_calls(name, calls, reps, flush, e0, e1, peaks):
    """Time each (fn, work, unit) of `calls` alone: median of `reps` CUDA-event timings,
    L2 flushed before each; print one JSON line per kernel."""
    for kname, (fn, work, unit) in calls.items():
        for _ in range(3):
            fn()
        times = []
        for _ in range(reps):
            flush.zero_()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        rate = work / (ms * 1e-3) / scale
        best = work / (min(times) * 1e-3) / scale
        peak = peaks["bf16_tflops"] if unit == "TFLOP/s" else peaks["hbm_gbs"]
        rec = {"workload": name, "kernel": kname, "ms": ms, "rate": rate, "unit": unit,
               "frac_of_measured_peak": rate / peak, "best_ms": min(times), "best_rate": best, "reps": reps,
               "l2": "flushed before each call"}
        if unit == "TFLOP/s" and peaks.get("bf16_tflops_sustained"):
            rec["frac_of_sustained_peak"] = rate / peaks["bf16_tflops_sustained"]
        print(json.dumps(rec))


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES), help="run one kernel on a reduced case (for ncu)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--all-workloads", action="store_true",
                    help="time every named workload's kernels alone (one JSON line each)")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the float64 oracle (dense, block-tiled, row-wise) on every named workload")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args.profile, args.reps)
        return
    if args.all_workloads:
        run_all_workloads(max(args.reps, 20))
        return
    if args.oracle_configs:
        run_oracle_configs()
        return
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
