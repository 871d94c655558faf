"""Helpers for the GPU parity tests: library build/load, tensor conversion, error metrics."""
import numpy as np
import pytest
import torch

# Bars from the benchmark spec of the path (floating point, so within tolerance):
O_MAX_ABS = 1e-2        # forward O, max-abs over all elements
LSE_MAX_ABS = 2e-3      # LSE, max-abs over all rows
GRAD_REL_FRO = 2e-2     # dQ, dK, dV relative Frobenius error, each tensor
PRECISE_O_MAX_ABS = 1e-4  # fp32 O of the single-head N=256, d=64 forward on the precise path


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_attention_flash_gb300.build import build

    build()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


def rel_fro(got, ref) -> float:
    """||got - ref||_F / ||ref||_F; for an exactly zero reference (e.g. dQ and dK
    with a single key, where dS = P * (dP - D) vanishes) the absolute norm."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def bf16_half_ulp(x) -> np.ndarray:
    """Half a bf16 ulp at |x| (8 significant bits): the rounding error of storing x in bf16."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def o_within_bar(got, ref, out_dtype) -> float:
    """Largest excess of |got - ref| over the O bar: 1e-2 for fp32 output; for bf16
    output 1e-2 plus the storage rounding of bf16 at the reference value.
    Returns a value <= 0 when every element is within the bar."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    bar = O_MAX_ABS + (bf16_half_ulp(ref) if out_dtype == "bf16" else 0.0)
    return float(np.max(err - bar))
