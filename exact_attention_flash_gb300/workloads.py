"""Seeded synthetic inputs (no attention arithmetic here).

Every tensor is drawn i.i.d. N(0, 1) in float32 by a torch generator seeded
with the workload's seed, on the device the caller names, in the order
Q, K, V, dO, and rounded to bf16 (round to nearest even).  Where a workload
stresses large logits, Q and K are then multiplied by a power of two (exact
in bf16).  Large tensors are drawn in slices along the batch axis so the
float32 staging stays small; the slice order is fixed, so the values depend
only on the seed and the device type.

The same function feeds the CUDA path and the oracle: the oracle receives
float64 copies of the very bf16 values the kernels read.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str               # "attention" (forward, optionally backward) or "decode"
    B: int
    H: int
    N: int                  # query/key length (attention) or KV length (decode)
    d: int
    seed: int
    causal: bool = False
    backward: bool = False
    qk_mult: float = 1.0
    out_f32: bool = False   # forward output O in fp32 (else bf16)
    n_split: int = 0        # decode only

    @property
    def scale(self) -> float:
        return self.d ** -0.5


# The five measured shapes of exact attention on one GPU.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("fwd_b1h1_n256_d64", "attention", 1, 1, 256, 64, seed=0, out_f32=True),
        Workload("causal_fwdbwd_b4h16_n2048_d64", "attention", 4, 16, 2048, 64, seed=1, causal=True, backward=True),
        Workload("causal_fwdbwd_b2h16_n8192_d128_qk8", "attention", 2, 16, 8192, 128, seed=2, causal=True,
                 backward=True, qk_mult=8.0),
        Workload("fwd_b1h32_n16384_d128", "attention", 1, 32, 16384, 128, seed=3),
        Workload("decode_b16h32_l32768_d128_s64", "decode", 16, 32, 32768, 128, seed=4, n_split=64),
    ]
}


def _randn_bf16(shape, gen, device, slices=1):
    """N(0,1) float32 draws rounded to bf16; drawn in `slices` pieces along dim 0."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    step = max(1, shape[0] // slices)
    for i in range(0, shape[0], step):
        piece = torch.randn((min(step, shape[0] - i),) + tuple(shape[1:]), generator=gen, dtype=torch.float32,
                            device=device)
        out[i : i + piece.shape[0]] = piece.to(torch.bfloat16)
    return out


def make_attention_inputs(B, H, N, d, seed, device="cuda", qk_mult=1.0, with_do=True):
    """q, k, v (and dO) bf16 [B, H, N, d] for one seed."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    slices = B if B * H * N * d > (1 << 26) else 1
    q = _randn_bf16((B, H, N, d), gen, device, slices)
    k = _randn_bf16((B, H, N, d), gen, device, slices)
    v = _randn_bf16((B, H, N, d), gen, device, slices)
    do = _randn_bf16((B, H, N, d), gen, device, slices) if with_do else None
    if qk_mult != 1.0:
        q.mul_(qk_mult)
        k.mul_(qk_mult)
    return q, k, v, do


def make_decode_inputs(B, H, L, d, seed, device="cuda"):
    """q [B, H, 1, d] and k, v [B, H, L, d] bf16 for one seed."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn_bf16((B, H, 1, d), gen, device)
    k = _randn_bf16((B, H, L, d), gen, device, slices=B)
    v = _randn_bf16((B, H, L, d), gen, device, slices=B)
    return q, k, v


def make_inputs(w: Workload, device="cuda"):
    if w.kind == "decode":
        return make_decode_inputs(w.B, w.H, w.N, w.d, w.seed, device)
    return make_attention_inputs(w.B, w.H, w.N, w.d, w.seed, device, w.qk_mult, with_do=w.backward)
