"""The GPU parity suite once more, on the bounds-checked build.

compute-sanitizer is not available on this machine. In its place,
libfa_gb300_checked.so (the same sources compiled with FA_BOUNDS_CHECK) checks
every computed global access of every kernel against its buffer's extent:
- the O and LSE stores of the forward, and its key-major form's workspace accesses;
- the backward's preprocess loads and stores, bias-tile copies, dQ reductions and
  zero-gradient tiles;
- the decode's q, K and V loads, segment states and counters;
- the merge's rows.
A miss is recorded in a status word and the access is skipped, so nothing faults.
This test runs every other GPU test in a subprocess that loads the checked
library (FA_GB300_LIBRARY). Those tests check fa_device_status() == FA_OK after
their calls, so a single out-of-extent index anywhere fails them
(FA_ERR_BOUNDS). Their parity checks must pass as well.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


def test_gpu_suite_on_the_bounds_checked_build():
    require_gpu()
    from exact_attention_flash_gb300.build import build

    lib = build(checked=True)
    env = dict(os.environ, FA_GB300_LIBRARY=str(lib))
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "--ignore", str(Path(__file__).resolve()), str(ROOT / "tests")]
    res = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    tail = "\n".join(res.stdout.splitlines()[-15:])
    assert res.returncode == 0, tail + res.stderr[-2000:]
    assert " passed" in tail and "failed" not in tail
