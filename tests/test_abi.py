"""The C-ABI library builds, loads and exports every symbol its header declares;
host-side argument checks reject bad calls before any CUDA work (CPU only)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "fa_gb300.h"


@pytest.fixture(scope="module")
def lib():
    from exact_attention_flash_gb300 import _lib
    from exact_attention_flash_gb300.build import build

    build()
    return _lib.load()


def _declared():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("fa_forward", "fa_forward_workspace_size", "fa_backward", "fa_backward_workspace_size",
                     "fa_decode", "fa_decode_workspace_size", "fa_get_device_status", "fa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    from exact_attention_flash_gb300 import _lib

    for name in _declared():
        assert hasattr(lib, name), f"{name} not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_version_and_status_strings(lib):
    assert lib.fa_abi_version() == 3
    assert lib.fa_status_string(0) == b"ok"
    assert lib.fa_status_string(4) == b"device wait timed out"


def test_workspace_sizes(lib):
    # per query row (padded to a multiple of 64): two 32-byte rows of bias tiles
    assert lib.fa_backward_workspace_size(2, 16, 8192, 128, 1) == 2 * 16 * 8192 * 64
    assert lib.fa_backward_workspace_size(1, 1, 65, 64, 1) == 128 * 64  # rows padded to 128
    # bf16 gradients add the fp32 dQ accumulator after the bias tiles (256-byte aligned)
    assert lib.fa_backward_workspace_size(2, 16, 8192, 128, 0) == 2 * 16 * 8192 * 64 + 2 * 16 * 8192 * 128 * 4
    assert lib.fa_backward_workspace_size(1, 1, 65, 64, 0) == 8192 + 65 * 64 * 4
    assert lib.fa_backward_workspace_size(1, 1, 3, 64, 0) == 64 * 64 + 3 * 64 * 4
    assert lib.fa_backward_workspace_size(1, 1, 8, 64, 2) == 0
    counters = ((16 * 32 * 4 + 255) // 256) * 256
    partials = 16 * 32 * 64 * 130 * 4
    assert lib.fa_decode_workspace_size(16, 32, 128, 64) == counters + ((partials + 255) // 256) * 256
    assert lib.fa_decode_workspace_size(1, 1, 128, 0) == 0
    # the forward's workspace holds one work counter, padded to 256 bytes, for any size
    assert lib.fa_forward_workspace_size(2, 16, 8192, 128, 1) == 256
    assert lib.fa_forward_workspace_size(1, 1, 1, 64, 0) == 256
    assert lib.fa_forward_workspace_size(0, 1, 1, 64, 0) == 0


def test_decode_workspace_size_never_wraps(lib):
    # B, H <= 65535 and n_split <= 2^30 would make B * H * n_split * (d + 2) * 4 pass
    # 2^64: such sizes are reported as 0 (too large), never as a small wrapped value.
    assert lib.fa_decode_workspace_size(65535, 65535, 128, 1 << 30) == 0
    r256 = lambda x: ((x + 255) // 256) * 256  # noqa: E731
    heads = 65535 * 65535
    assert lib.fa_decode_workspace_size(65535, 65535, 64, 1 << 20) == r256(heads * 4) + r256(heads * (1 << 20) * 264)
    assert lib.fa_decode_workspace_size(65535, 65535, 128, 1 << 24) == 0  # 2^24 * 520 * heads > 2^62
    big = lib.fa_decode_workspace_size(65535, 65535, 128, 64)
    assert big == ((65535 * 65535 * 4 + 255) // 256) * 256 + ((65535 * 65535 * 64 * 130 * 4 + 255) // 256) * 256


FAKE = 1 << 20  # a non-null, aligned pointer value; never dereferenced on these paths


WS = (FAKE, 256)  # a forward workspace argument pair that passes the checks


def test_forward_rejects_bad_arguments(lib):
    # fa_forward(q, k, v, o, o_dtype, lse, B, H, N, d, scale, causal, precise, workspace, bytes, stream)
    assert lib.fa_forward(None, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, 0, *WS, None) == 1
    assert lib.fa_forward(FAKE + 2, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, 0, *WS, None) == 1
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 7, FAKE, 1, 1, 8, 64, 0.0, 0, 0, *WS, None) == 1
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 0, 64, 0.0, 0, 0, *WS, None) == 1
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 96, 0.0, 0, 0, *WS, None) == 2
    # the workspace: missing, too small, misaligned
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, 0, None, 256, None) == 5
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, 0, FAKE, 255, None) == 5
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, 0, FAKE + 4, 256, None) == 5


def test_backward_rejects_bad_arguments(lib):
    # fa_backward(q, k, v, o, o_dtype, lse, dout, dq, dk, dv, grad_dtype, B, H, N, d, scale, causal, ws, bytes, stream)
    args = [FAKE] * 4 + [0, FAKE, FAKE, FAKE, FAKE, FAKE]
    assert lib.fa_backward(*args, 1, 1, 1, 8, 80, 0.0, 1, FAKE, 1 << 20, None) == 2
    assert lib.fa_backward(*args, 1, 1, 1, 8, 64, 0.0, 1, FAKE, 4, None) == 5
    assert lib.fa_backward(*args, 1, 1, 1, 8, 64, 0.0, 1, None, 1 << 20, None) == 5
    assert lib.fa_backward(*args, 5, 1, 1, 8, 64, 0.0, 1, FAKE, 1 << 20, None) == 1  # grad_dtype
    # bf16 gradients need the larger workspace: the fp32-gradient size is too small
    small = lib.fa_backward_workspace_size(1, 1, 64, 64, 1)
    assert lib.fa_backward(*args, 0, 1, 1, 64, 64, 0.0, 1, FAKE, small, None) == 5


def test_decode_rejects_bad_arguments(lib):
    ws = 1 << 24
    # n_split < 1 is an error, as the page's flash_decode raises on it.
    assert lib.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0.0, 0, None, FAKE, ws, None) == 1
    assert lib.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 0, 128, 0.0, 4, None, FAKE, ws, None) == 1
    assert lib.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 32, 0.0, 4, None, FAKE, ws, None) == 2
    assert lib.fa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 128, 0.0, 4, None, FAKE, 8, None) == 5
    assert lib.fa_debug_wait_timeout(0, None) == 1


def test_offset_entry_points_reject_bad_arguments(lib):
    # fa_forward_qk(q, k, v, o, o_dtype, lse, B, H, Nq, Nk, q_start, d, scale, causal, precise, ws, bytes, stream)
    assert lib.fa_forward_qk(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 16, -1, 64, 0.0, 1, 0, *WS, None) == 1
    assert lib.fa_forward_qk(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 0, 0, 64, 0.0, 1, 0, *WS, None) == 1
    assert lib.fa_forward_qk(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 16, 2**31 - 4, 64, 0.0, 1, 0, *WS, None) == 1
    assert lib.fa_forward_qk(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 16, 0, 48, 0.0, 1, 0, *WS, None) == 2
    assert lib.fa_forward_qk(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 16, 0, 64, 0.0, 1, 0, FAKE, 8, None) == 5
    args = [FAKE] * 4 + [0, FAKE, FAKE, FAKE, FAKE, FAKE, 1]
    # fa_backward_qk(..., grad_dtype, B, H, Nq, Nk, q_start, d, scale, causal, workspace, bytes, stream)
    assert lib.fa_backward_qk(*args, 1, 1, 8, 16, -3, 64, 0.0, 1, FAKE, 1 << 20, None) == 1
    assert lib.fa_backward_qk(*args, 1, 1, 8, 0, 0, 64, 0.0, 1, FAKE, 1 << 20, None) == 1
    assert lib.fa_backward_qk(*args, 1, 1, 8, 16, 0, 64, 0.0, 1, FAKE, 4, None) == 5


def test_counts_beyond_32_bits_are_unsupported(lib):
    # B * H = 2^31 heads; then 2^30 heads whose forward items (ceil(1024 / 256) each)
    # or backward CTAs (ceil(1024 / 128) each) pass 2^31: rejected before any CUDA call
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1 << 16, 1 << 15, 8, 64, 0.0, 0, 0, *WS, None) == 2
    assert lib.fa_forward(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1 << 20, 1 << 10, 1024, 64, 0.0, 0, 0, *WS, None) == 2
    args = [FAKE] * 4 + [0, FAKE, FAKE, FAKE, FAKE, FAKE, 1]
    assert lib.fa_backward(*args, 1 << 20, 1 << 10, 1024, 64, 0.0, 0, FAKE, 1 << 62, None) == 2


def test_merge_and_auto_split_reject_bad_arguments(lib):
    # fa_merge_states(o_a, lse_a, o_b, lse_b, o, lse, o_dtype, rows, d, stream)
    assert lib.fa_merge_states(None, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 128, None) == 1
    assert lib.fa_merge_states(FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 128, None) == 1
    assert lib.fa_merge_states(FAKE, FAKE + 2, FAKE, FAKE, FAKE, FAKE, 1, 4, 128, None) == 1
    assert lib.fa_merge_states(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 126, None) == 1
    assert lib.fa_merge_states(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 4, 128, None) == 1
    assert lib.fa_merge_states(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, -1, 128, None) == 1
    assert lib.fa_merge_states(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 128, None) == 0  # nothing to do
    assert lib.fa_decode_auto_split(0, 1, 100) == 0
    assert lib.fa_decode_auto_split(1, 1, 0) == 0


def test_keymajor_workspace_and_arguments(lib):
    rows = 2 * 3 * 100
    assert lib.fa_forward_keymajor_workspace_size(2, 3, 100, 128) == ((rows * 128 * 4 + 255) // 256 + 2 * ((rows * 4 + 255) // 256)) * 256
    assert lib.fa_forward_keymajor_workspace_size(0, 3, 100, 128) == 0
    # (q, k, v, o, o_dtype, lse, B, H, N, d, scale, causal, workspace, bytes, stream)
    assert lib.fa_forward_keymajor(None, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, FAKE, 1 << 20, None) == 1
    assert lib.fa_forward_keymajor(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 48, 0.0, 0, FAKE, 1 << 20, None) == 2
    assert lib.fa_forward_keymajor(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 1, 8, 64, 0.0, 0, FAKE, 16, None) == 5


def test_set_stats_arguments(lib):
    # the counters must be 8-byte aligned; NULL stops counting (nothing runs here)
    assert lib.fa_set_stats(FAKE + 4) == 1
    assert lib.fa_set_stats(FAKE) == 0
    assert lib.fa_set_stats(None) == 0


def test_python_layer_fails_loudly_without_library(monkeypatch, tmp_path):
    from exact_attention_flash_gb300 import _lib

    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()
