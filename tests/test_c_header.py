"""include/fa_gb300.h as a C interface (CPU only).

A C99 program, and the same source compiled as C++, includes the header. It links
libfa_gb300.so with the system toolchain and checks, without a GPU:
- the version;
- the status strings;
- the workspace sizes;
- argument errors: each entry point rejects a bad argument synchronously, before
  any CUDA call.
This is the boundary a caller without Python uses.
"""
import shutil
import subprocess

import pytest

from tests.test_abi import HEADER, ROOT

PROGRAM = r"""
#include "fa_gb300.h"
#include <stdio.h>
#include <string.h>

static int failures = 0;
#define CHECK(cond) do { if (!(cond)) { printf("failed: %s (line %d)\n", #cond, __LINE__); ++failures; } } while (0)

int main(void) {
  void* p = (void*)(size_t)4096;          /* aligned, never dereferenced: every call below fails its checks first */
  float* f = (float*)p;
  char ws_small[16];
  CHECK(fa_abi_version() == FA_ABI_VERSION);
  CHECK(strcmp(fa_status_string(FA_OK), "ok") == 0);
  CHECK(fa_status_string(FA_ERR_WORKSPACE) != NULL);
  CHECK(fa_backward_workspace_size(2, 16, 8192, 128, FA_F32) == (size_t)2 * 16 * 8192 * 64);
  CHECK(fa_backward_workspace_size(2, 16, 8192, 128, FA_BF16) ==
        (size_t)2 * 16 * 8192 * 64 + (size_t)2 * 16 * 8192 * 128 * 4);
  CHECK(fa_backward_workspace_size(0, 16, 8192, 128, FA_F32) == 0);
  CHECK(fa_decode_workspace_size(16, 32, 128, 64) > 0);
  CHECK(fa_decode_auto_split(0, 32, 32768) == 0);
  /* argument errors */
  CHECK(fa_forward_workspace_size(2, 16, 8192, 128, 1) == 256);
  CHECK(fa_forward(NULL, p, p, p, FA_BF16, f, 1, 1, 8, 64, 0.f, 0, 0, p, 256, NULL) == FA_ERR_INVALID_ARG);
  CHECK(fa_forward(p, p, p, p, FA_BF16, f, 1, 1, 8, 96, 0.f, 0, 0, p, 256, NULL) == FA_ERR_UNSUPPORTED);
  CHECK(fa_forward(p, p, p, p, FA_BF16, f, 1, 1, 8, 64, 0.f, 0, 0, ws_small, sizeof ws_small, NULL) ==
        FA_ERR_WORKSPACE);
  CHECK(fa_forward_qk(p, p, p, p, FA_BF16, f, 1, 1, 8, 16, -1, 64, 0.f, 1, 0, p, 256, NULL) == FA_ERR_INVALID_ARG);
  CHECK(fa_backward(p, p, p, p, FA_BF16, f, p, p, p, p, (fa_dtype)7, 1, 1, 8, 64, 0.f, 1, p, 1u << 20, NULL) ==
        FA_ERR_INVALID_ARG);
  CHECK(fa_backward(p, p, p, p, FA_BF16, f, p, p, p, p, FA_BF16, 1, 1, 8, 64, 0.f, 1, ws_small, sizeof ws_small,
                    NULL) == FA_ERR_WORKSPACE);
  CHECK(fa_decode(p, p, p, f, f, 1, 1, 16, 128, 0.f, 0, NULL, p, 1u << 20, NULL) == FA_ERR_INVALID_ARG);
  CHECK(fa_merge_states(NULL, f, p, f, p, f, FA_F32, 4, 128, NULL) == FA_ERR_INVALID_ARG);
  CHECK(fa_set_stats((unsigned long long*)(size_t)4100) == FA_ERR_INVALID_ARG);  /* counters must be 8-byte aligned */
  printf("%d failures\n", failures);
  return failures != 0;
}
"""


def _compile_and_run(tmp_path, compiler, std, ext):
    from exact_attention_flash_gb300.build import LIB, build

    build()
    src = tmp_path / f"abi_check.{ext}"
    src.write_text(PROGRAM)
    exe = tmp_path / f"abi_check_{ext}"
    cmd = [compiler, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", str(HEADER.parent), str(src),
           "-o", str(exe), "-L", str(LIB.parent), "-l:" + LIB.name, f"-Wl,-rpath,{LIB.parent}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "0 failures" in run.stdout


@pytest.mark.parametrize("compiler,std,ext", [("gcc", "c99", "c"), ("g++", "c++17", "cpp")])
def test_header_compiles_and_links_as_c_and_cpp(tmp_path, compiler, std, ext):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not available")
    _compile_and_run(tmp_path, compiler, std, ext)


def test_program_covers_every_error_code():
    for code in ("FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_WORKSPACE"):
        assert code in PROGRAM
    assert (ROOT / "include" / "fa_gb300.h").exists()
