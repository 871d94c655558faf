"""Build the sm_103a shared library ``libfa_gb300.so`` in-tree with nvcc.

Each ``csrc/*.cu`` file is compiled in parallel to an object under ``_build/``
and the objects are linked into one shared library next to this file.  Objects
are rebuilt when their source or any header is newer.

``build(checked=True)`` builds the same sources with ``FA_BOUNDS_CHECK`` into
``libfa_gb300_checked.so`` (objects under ``_build_checked/``): every computed
global access then checks its index against its buffer's extent and reports a
miss through ``fa_device_status()`` as FA_ERR_BOUNDS.  Load it by setting
``FA_GB300_LIBRARY`` to its path before importing the package.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
BUILD = PKG / "_build"
LIB = PKG / "libfa_gb300.so"
BUILD_CHECKED = PKG / "_build_checked"
LIB_CHECKED = PKG / "libfa_gb300_checked.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--use_fast_math", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")
    return cand


def _compile(nvcc: str, src: Path, headers_mtime: float, out_dir: Path, extra: list[str]) -> tuple[Path, str]:
    obj = out_dir / (src.stem + ".o")
    if obj.exists() and obj.stat().st_mtime >= max(src.stat().st_mtime, headers_mtime):
        return obj, ""
    cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", str(INCLUDE), "-c", str(src), "-o", str(obj)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def build(verbose: bool = False, checked: bool = False) -> Path:
    nvcc = _nvcc()
    out_dir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    extra = ["-DFA_BOUNDS_CHECK"] if checked else []
    out_dir.mkdir(exist_ok=True)
    headers = list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + list(INCLUDE.glob("*.h"))
    headers_mtime = max((h.stat().st_mtime for h in headers), default=0.0)
    sources = sorted(CSRC.glob("*.cu"))
    with cf.ThreadPoolExecutor(max_workers=min(len(sources), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, headers_mtime, out_dir, extra), sources))
    objs = [r[0] for r in results]
    if verbose:
        for _, log in results:
            if log:
                print(log)
    newest = max(o.stat().st_mtime for o in objs)
    if not lib_path.exists() or lib_path.stat().st_mtime < newest:
        tmp = lib_path.with_suffix(".so.tmp")
        cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-lcudart"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True))
