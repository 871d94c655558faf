"""GB300-native exact tiled attention: forward, recompute backward, split-KV decode.

The Python layer only marshals arguments: torch allocates device memory and
supplies the stream, and every step of the computation runs in the sm_103a
kernels of ``libfa_gb300.so`` reached through its C ABI (``include/fa_gb300.h``).
"""
from __future__ import annotations

import contextlib
import functools

import torch

from . import _lib
from ._lib import FAError

__all__ = ["flash_attention", "fa_forward", "fa_backward", "fa_decode", "fa_device_status", "fa_get_device_status",
           "FAError", "forward_workspace_bytes", "backward_workspace_bytes",
           "decode_workspace_bytes", "fa_set_stats", "stats_counters", "STATS_FIELDS", "fa_merge_states",
           "decode_auto_split", "fa_forward_keymajor"]

# Order of the counters behind fa_set_stats ("attention_kernels.py" sections 3-4, ``stats``).
STATS_FIELDS = ("tiles", "skipped", "rescales", "dq_atomic_adds")


def _on_tensor_device(fn):
    """Make the first argument's GPU the current device for the call, so that the
    library launches there and on that device's current stream."""
    @functools.wraps(fn)
    def wrapper(t, *args, **kwargs):
        if not (isinstance(t, torch.Tensor) and t.is_cuda):
            return fn(t, *args, **kwargs)  # the argument checks raise
        others = [a for a in list(args) + list(kwargs.values()) if isinstance(a, torch.Tensor)]
        if any(a.device != t.device for a in others):
            raise ValueError(f"{fn.__name__}: every tensor must be on {t.device}")
        with torch.cuda.device(t.device):
            return fn(t, *args, **kwargs)
    return wrapper


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_bf16(name, t, shape=None):
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _scale_arg(scale):
    return 0.0 if scale is None else float(scale)


def _check_workspace(t):
    if not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor")


def _check_out(name, t, shape, dtypes):
    if not t.is_cuda or t.dtype not in dtypes or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous CUDA tensor of shape {tuple(shape)} and dtype in {dtypes}")


def forward_workspace_bytes(B, H, N, d, causal=False) -> int:
    """Workspace bytes of :func:`fa_forward` (the persistent grid's work counter)."""
    return int(_lib.load().fa_forward_workspace_size(B, H, N, d, int(bool(causal))))


@_on_tensor_device
def fa_forward(q, k, v, causal=False, scale=None, out_dtype=torch.bfloat16, precise=False, out=None, lse=None,
               stream=None, q_start=0, workspace=None):
    """O, LSE = softmax(Q K^T * scale [causal]) V.

    q [B, H, Nq, d], k and v [B, H, Nk, d], bf16.  Query row i sits at position
    q_start + i; with ``causal`` it sees the keys j <= q_start + i.  Nq = Nk with
    q_start = 0 is ordinary self-attention.  ``workspace``: a uint8 CUDA tensor of
    at least :func:`forward_workspace_bytes`; one is allocated when None.  Calls
    whose GPU work overlaps (other streams, graphs replayed at once) need
    workspaces of their own.
    """
    lib = _lib.load()
    _check_bf16("q", q)
    B, H, Nq, d = q.shape
    if k.dim() != 4:
        raise ValueError("k must be [B, H, Nk, d]")
    Nk = k.shape[2]
    _check_bf16("k", k, (B, H, Nk, d))
    _check_bf16("v", v, (B, H, Nk, d))
    if out is None:
        out = torch.empty((B, H, Nq, d), device=q.device, dtype=out_dtype)
    _check_out("out", out, (B, H, Nq, d), (torch.bfloat16, torch.float32))
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    _check_out("lse", lse, (B, H, Nq), (torch.float32,))
    if workspace is None:
        workspace = torch.empty(forward_workspace_bytes(B, H, Nq, d, causal), device=q.device, dtype=torch.uint8)
    _check_workspace(workspace)
    o_code = _lib.FA_F32 if out.dtype == torch.float32 else _lib.FA_BF16
    code = lib.fa_forward_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), o_code, lse.data_ptr(),
                             B, H, Nq, Nk, int(q_start), d, _scale_arg(scale), int(bool(causal)), int(bool(precise)),
                             workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _lib.check("fa_forward_qk", code)
    return out, lse


def backward_workspace_bytes(B, H, N, d, grad_dtype=torch.float32) -> int:
    """Workspace bytes of :func:`fa_backward` (N = Nq) for gradients of ``grad_dtype``."""
    return int(_lib.load().fa_backward_workspace_size(B, H, N, d, _grad_code(grad_dtype)))


def _grad_code(grad_dtype):
    if grad_dtype == torch.float32:
        return _lib.FA_F32
    if grad_dtype == torch.bfloat16:
        return _lib.FA_BF16
    raise ValueError("grad_dtype must be torch.float32 or torch.bfloat16")


@_on_tensor_device
def fa_backward(q, k, v, o, lse, do, causal=False, scale=None, workspace=None, dq=None, dk=None, dv=None,
                stream=None, q_start=0, grad_dtype=torch.float32):
    """dQ, dK, dV of sum(O * dO) by recomputation from LSE.

    Shapes as for :func:`fa_forward` (q, o, do [B, H, Nq, d]; k, v [B, H, Nk, d];
    lse [B, H, Nq]); causal, scale and q_start must match the forward call.  The
    products accumulate in fp32; ``grad_dtype`` (fp32 or bf16) is the type of the
    returned gradients.
    """
    lib = _lib.load()
    g_code = _grad_code(grad_dtype)
    _check_bf16("q", q)
    B, H, Nq, d = q.shape
    if k.dim() != 4:
        raise ValueError("k must be [B, H, Nk, d]")
    Nk = k.shape[2]
    _check_bf16("k", k, (B, H, Nk, d))
    _check_bf16("v", v, (B, H, Nk, d))
    _check_bf16("do", do, q.shape)
    _check_out("o", o, q.shape, (torch.bfloat16, torch.float32))
    _check_out("lse", lse, (B, H, Nq), (torch.float32,))
    nbytes = backward_workspace_bytes(B, H, Nq, d, grad_dtype)
    if workspace is None:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    dq = torch.empty((B, H, Nq, d), device=q.device, dtype=grad_dtype) if dq is None else dq
    dk = torch.empty((B, H, Nk, d), device=q.device, dtype=grad_dtype) if dk is None else dk
    dv = torch.empty((B, H, Nk, d), device=q.device, dtype=grad_dtype) if dv is None else dv
    _check_out("dq", dq, (B, H, Nq, d), (grad_dtype,))
    _check_out("dk", dk, (B, H, Nk, d), (grad_dtype,))
    _check_out("dv", dv, (B, H, Nk, d), (grad_dtype,))
    o_code = _lib.FA_F32 if o.dtype == torch.float32 else _lib.FA_BF16
    code = lib.fa_backward_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), o_code, lse.data_ptr(),
                              do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), g_code, B, H, Nq, Nk,
                              int(q_start), d, _scale_arg(scale), int(bool(causal)), workspace.data_ptr(),
                              workspace.numel(), _stream_ptr(stream))
    _lib.check("fa_backward_qk", code)
    return dq, dk, dv


def decode_workspace_bytes(B, H, d, n_split) -> int:
    return int(_lib.load().fa_decode_workspace_size(B, H, d, n_split))


def decode_auto_split(B, H, L) -> int:
    """The library's split count for B * H heads of L keys on the current device."""
    n = int(_lib.load().fa_decode_auto_split(B, H, L))
    if n < 1:
        raise ValueError("fa_decode_auto_split: bad sizes or no device")
    return n


@_on_tensor_device
def fa_decode(q, k, v, n_split=None, scale=None, return_partials=False, workspace=None, out=None, lse=None,
              stream=None):
    """Split-KV decode: q [B, H, 1, d], k/v [B, H, L, d] bf16 -> O [B, H, 1, d] fp32, LSE [B, H].

    ``n_split=None`` takes :func:`decode_auto_split`'s count.
    """
    lib = _lib.load()
    _check_bf16("q", q)
    _check_bf16("k", k)
    _check_bf16("v", v, k.shape)
    B, H, L, d = k.shape
    if tuple(q.shape) != (B, H, 1, d):
        raise ValueError("q must be [B, H, 1, d]")
    if n_split is None:
        n_split = decode_auto_split(B, H, L)
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(B, H, d, max(int(n_split), 1)), device=q.device,
                                dtype=torch.uint8)
    out = torch.empty((B, H, 1, d), device=q.device, dtype=torch.float32) if out is None else out
    lse = torch.empty((B, H), device=q.device, dtype=torch.float32) if lse is None else lse
    _check_out("out", out, (B, H, 1, d), (torch.float32,))
    _check_out("lse", lse, (B, H), (torch.float32,))
    parts = None
    if return_partials:
        parts = torch.empty((B, H, max(int(n_split), 1), d + 2), device=q.device, dtype=torch.float32)
    code = lib.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, L, d,
                         _scale_arg(scale), int(n_split), 0 if parts is None else parts.data_ptr(),
                         workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _lib.check("fa_decode", code)
    return (out, lse, parts) if return_partials else (out, lse)


def fa_get_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the kernels' device status as an fa_status code."""
    return int(_lib.load().fa_get_device_status(_stream_ptr(stream)))


fa_device_status = fa_get_device_status


def fa_set_stats(counters=None) -> None:
    """Count the page's ``stats`` for the fa_forward / fa_backward calls this host thread makes.

    ``counters``: a CUDA int64 tensor of 4 elements (zeroed by the caller), which
    the kernels add into in the order of ``STATS_FIELDS``; None stops counting.
    See ``fa_set_stats`` in ``include/fa_gb300.h`` for what each counter holds.
    """
    if counters is None:
        ptr = None
    else:
        if not counters.is_cuda or counters.dtype != torch.int64 or counters.numel() != 4 or not counters.is_contiguous():
            raise ValueError("counters must be a contiguous CUDA int64 tensor of 4 elements")
        ptr = counters.data_ptr()
    _lib.check("fa_set_stats", _lib.load().fa_set_stats(ptr))


@contextlib.contextmanager
def stats_counters(device=None):
    """Zeroed counters set for the calls inside the ``with`` block; yields the tensor."""
    c = torch.zeros(4, dtype=torch.int64, device=device or "cuda")
    fa_set_stats(c)
    try:
        yield c
    finally:
        fa_set_stats(None)


@_on_tensor_device
def fa_merge_states(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """Merge two attention results over disjoint key sets ("attention_kernels.py" section 1 ``merge_states``).

    o_a, o_b: [..., d] fp32 or bf16 (one shape and dtype); lse_a, lse_b: [...] fp32.
    Returns (O, LSE) of the attention over both key sets; ``out`` and ``lse`` may
    be the inputs (in place).
    """
    lib = _lib.load()
    if o_a.dtype != o_b.dtype or o_a.dtype not in (torch.float32, torch.bfloat16) or o_a.shape != o_b.shape:
        raise ValueError("o_a and o_b must have one shape and dtype (fp32 or bf16)")
    d = o_a.shape[-1]
    lead = tuple(o_a.shape[:-1])
    for name, t in (("o_a", o_a), ("o_b", o_b)):
        _check_out(name, t, o_a.shape, (o_a.dtype,))
    for name, t in (("lse_a", lse_a), ("lse_b", lse_b)):
        _check_out(name, t, lead, (torch.float32,))
    out = torch.empty_like(o_a) if out is None else out
    lse = torch.empty_like(lse_a) if lse is None else lse
    _check_out("out", out, o_a.shape, (o_a.dtype,))
    _check_out("lse", lse, lead, (torch.float32,))
    code = lib.fa_merge_states(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(), lse_b.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), _lib.FA_F32 if o_a.dtype == torch.float32 else _lib.FA_BF16,
                               lse_a.numel(), d, _stream_ptr(stream))
    _lib.check("fa_merge_states", code)
    return out, lse


@_on_tensor_device
def fa_forward_keymajor(q, k, v, causal=False, scale=None, out_dtype=torch.bfloat16, workspace=None, stream=None):
    """O, LSE as :func:`fa_forward` gives them, computed in the first algorithm's key-major loop order.

    For comparison only: one CTA per (batch, head), much slower than fa_forward.
    q, k, v [B, H, N, d] bf16.
    """
    lib = _lib.load()
    _check_bf16("q", q)
    B, H, N, d = q.shape
    _check_bf16("k", k, q.shape)
    _check_bf16("v", v, q.shape)
    out = torch.empty((B, H, N, d), device=q.device, dtype=out_dtype)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    nbytes = int(lib.fa_forward_keymajor_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    code = lib.fa_forward_keymajor(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   _lib.FA_F32 if out.dtype == torch.float32 else _lib.FA_BF16, lse.data_ptr(),
                                   B, H, N, d, _scale_arg(scale), int(bool(causal)), workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(stream))
    _lib.check("fa_forward_keymajor", code)
    return out, lse


class _FlashAttention(torch.autograd.Function):
    """fa_forward as the forward of an autograd node and fa_backward as its backward.

    The node saves Q, K, V, O and LSE. Its backward recomputes P from LSE, as the
    page's backward does. Autograd wants gradients in the inputs' dtype, so the
    gradients come back as bf16; every product still accumulates in fp32.
    """

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, q_start):
        o, lse = fa_forward(q, k, v, causal=causal, scale=scale, q_start=q_start)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.q_start = causal, scale, q_start
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = fa_backward(q, k, v, o, lse, do.to(torch.bfloat16).contiguous(), causal=ctx.causal,
                                 scale=ctx.scale, q_start=ctx.q_start, grad_dtype=torch.bfloat16)
        return dq, dk, dv, None, None, None


def flash_attention(q, k, v, causal=False, scale=None, q_start=0):
    """Differentiable O = softmax(Q K^T * scale [causal]) V for PyTorch training code.

    q [B, H, Nq, d], k and v [B, H, Nk, d], contiguous bf16 CUDA tensors; returns O
    [B, H, Nq, d] bf16.  Calling ``backward`` on anything computed from O runs
    fa_backward and leaves bf16 gradients in ``q.grad``, ``k.grad`` and ``v.grad``.
    """
    return _FlashAttention.apply(q, k, v, bool(causal), scale, int(q_start))
