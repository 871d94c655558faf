"""The bounds-checked build (CPU only).

The same sources compiled with FA_BOUNDS_CHECK make libfa_gb300_checked.so. In it,
every computed global access checks its index against its buffer's extent, and
fa_device_status() reports a miss as FA_ERR_BOUNDS. This test checks that:
- the checked library builds and exports every symbol the header declares;
- FA_GB300_LIBRARY selects it;
- its host-side argument checks answer as the normal build's do.
Running kernels through it is a GPU test (test_gpu_bounds_checked.py).
"""
import os
import subprocess
import sys

from tests.test_abi import ROOT, _declared

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
from exact_attention_flash_gb300 import _lib
lib = _lib.load()
assert _lib.LIB_PATH.name == "libfa_gb300_checked.so", _lib.LIB_PATH
for name in {names!r}:
    assert hasattr(lib, name), name
assert lib.fa_status_string(6) == b"index outside its buffer (bounds-checked build)"
assert lib.fa_backward_workspace_size(2, 16, 8192, 128, 1) == 2 * 16 * 8192 * 64
assert lib.fa_forward(None, 64, 64, 64, 0, 64, 1, 1, 8, 64, 0.0, 0, 0, 64, 256, None) == 1
print("ok")
"""


def test_checked_library_builds_exports_and_loads():
    from exact_attention_flash_gb300.build import LIB_CHECKED, build

    path = build(checked=True)
    assert path == LIB_CHECKED and path.exists()
    env = dict(os.environ, FA_GB300_LIBRARY=str(path))
    res = subprocess.run([sys.executable, "-c", SCRIPT.format(root=str(ROOT), names=_declared())], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout + res.stderr


def test_status_names_cover_the_header():
    from exact_attention_flash_gb300 import _lib

    header = (ROOT / "include" / "fa_gb300.h").read_text()
    for code, name in _lib.STATUS_NAMES.items():
        assert f"{name} = {code}" in header
