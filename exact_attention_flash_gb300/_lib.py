"""ctypes loader for ``libfa_gb300.so`` and the C-ABI signatures of ``include/fa_gb300.h``.

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``exact_attention_flash_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import os

# The library to load: the in-tree build, or another build of the same sources named
# by FA_GB300_LIBRARY (the bounds-checked one, libfa_gb300_checked.so).
LIB_PATH = Path(os.environ["FA_GB300_LIBRARY"]) if os.environ.get("FA_GB300_LIBRARY") else (
    Path(__file__).resolve().parent / "libfa_gb300.so")

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_CUDA",
    4: "FA_ERR_TIMEOUT",
    5: "FA_ERR_WORKSPACE",
    6: "FA_ERR_BOUNDS",
}
FA_BF16 = 0
FA_F32 = 1

# Every function the header declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t
SIGNATURES = {
    "fa_abi_version": (_I, []),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_forward_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "fa_forward": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_forward_qk": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_backward_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "fa_backward_qk": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "fa_backward": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "fa_decode_workspace_size": (_Z, [_I, _I, _I, _I]),
    "fa_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _Z, _P]),
    "fa_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    "fa_get_device_status": (_I, [_P]),
    "fa_device_status": (_I, [_P]),
    "fa_set_stats": (_I, [_P]),
    "fa_merge_states": (_I, [_P, _P, _P, _P, _P, _P, _I, ctypes.c_longlong, _I, _P]),
    "fa_forward_keymajor_workspace_size": (_Z, [_I, _I, _I, _I]),
    "fa_forward_keymajor": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "fa_decode_auto_split": (_I, [_I, _I, _I]),
    "fa_debug_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "fa_debug_abort_next_call": (_I, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


def load() -> ctypes.CDLL:
    """Load the library once; raise if it is not built."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"{LIB_PATH.name} is not built; run exact_attention_flash_gb300.build.build() (needs nvcc)"
            )
        lib = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(fn: str, code: int) -> None:
    if code != FA_OK:
        raise FAError(fn, code)
