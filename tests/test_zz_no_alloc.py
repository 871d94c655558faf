"""fa_decode_noalloc: split-KV decode for callers that cannot allocate device
memory or pass a workspace (for example a plugin handed no workspace by the
framework that owns the memory).  Its scratch is a fixed array inside the
library.  These tests call it through the C ABI and compare it with fa_decode,
which uses a caller-supplied workspace.  The file sorts last so a run that stops
at the first failure has run everything else first."""
import ctypes

import pytest
import torch

from tests.gpu_util import LSE_MAX_ABS, O_MAX_ABS, f64, max_abs, require_gpu

FAKE = 1 << 20  # aligned non-null pointer value; the size check returns before any CUDA call


def _lib():
    from exact_attention_flash_gb300 import _lib
    from exact_attention_flash_gb300.build import build

    build()
    return _lib.load()


CAP = 16 << 20  # FA_DECODE_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = _lib()
    # 16 x 32 heads x 64 segments x (128 + 2) floats is about 17 MB: more than the 16 MiB array.
    code = lib.fa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 32, 32768, 128, 0.0, 64, None, None)
    assert code == 5  # FA_ERR_WORKSPACE
    assert lib.fa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0.0, 0, None, None) == 1


def test_noalloc_limit_is_the_documented_workspace_size():
    """The check compares fa_decode_workspace_size() itself with the array's size:
    one segment more than the largest request that fits is refused with
    FA_ERR_WORKSPACE, before any CUDA call.  (The GPU test below runs the request
    of exactly the cap.)"""
    lib = _lib()
    # One head, d = 64: 256 bytes of counters plus 66 floats per segment state,
    # rounded up to 256 bytes.
    n_fit = max(n for n in range(60000, 70000) if lib.fa_decode_workspace_size(1, 1, 64, n) <= CAP)
    assert lib.fa_decode_workspace_size(1, 1, 64, n_fit) == CAP
    assert lib.fa_decode_workspace_size(1, 1, 64, n_fit + 1) > CAP
    assert lib.fa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 64, 0.0, n_fit + 1, None, None) == 5


def test_noalloc_huge_requests_are_refused_without_wrapping():
    """B, H and n_split near their limits: the size is never computed modulo 2^64,
    so no wrapped small value can pass the cap; the call is refused before any
    CUDA work."""
    lib = _lib()
    for B, H, n_split in [(65535, 65535, 1 << 30), (65535, 65535, 1 << 20), (65535, 65535, 64), (1, 1, 1 << 30)]:
        code = lib.fa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, 1 << 20, 128, 0.0, n_split, None, None)
        assert code in (2, 5), (B, H, n_split, code)  # FA_ERR_UNSUPPORTED (beyond 2^62) or FA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    require_gpu()
    lib = _lib()
    from exact_attention_flash_gb300 import fa_decode, fa_device_status
    from exact_attention_flash_gb300.workloads import make_decode_inputs

    stream = torch.cuda.current_stream().cuda_stream
    # Two calls in a row on the same shape (the second finds the first one's
    # contents in the shared array), then one on another shape.
    # The last case needs exactly the whole array: one head, d = 64, as many segments
    # as fit (most of them empty, since they outnumber the keys).
    n_cap = max(n for n in range(60000, 70000) if lib.fa_decode_workspace_size(1, 1, 64, n) <= CAP)
    cases = [(2, 4, 3000, 128, 16, 31), (2, 4, 3000, 128, 16, 32), (3, 2, 777, 64, 5, 33),
             (1, 1, 5000, 64, n_cap, 34)]
    for B, H, L, d, n_split, seed in cases:
        q, k, v = make_decode_inputs(B, H, L, d, seed, "cuda")
        ref_o, ref_l, ref_parts = fa_decode(q, k, v, n_split, return_partials=True)
        o = torch.full((B, H, 1, d), float("nan"), device="cuda")
        lse = torch.full((B, H), float("nan"), device="cuda")
        parts = torch.full((B, H, n_split, d + 2), float("nan"), device="cuda")
        code = lib.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, L,
                                     d, ctypes.c_float(0.0), n_split, parts.data_ptr(), stream)
        assert code == 0
        torch.cuda.synchronize()
        assert fa_device_status() == 0
        assert max_abs(f64(o), f64(ref_o)) <= O_MAX_ABS
        assert max_abs(f64(lse), f64(ref_l)) <= LSE_MAX_ABS
        assert max_abs(f64(parts[..., 2:]), f64(ref_parts[..., 2:])) <= O_MAX_ABS
