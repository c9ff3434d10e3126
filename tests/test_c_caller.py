"""The C ABI from a plain C program (no GPU): include/attn_fa2.h compiles as
C89 and C99, and a C caller linked against libattn_fa2.so gets the documented
statuses and messages from calls that are rejected before any CUDA work."""

import os
import shutil
import subprocess

import pytest


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "attn_fa2.h"

int main(void) {
  size_t bytes = 0;
  int st;
  /* workspace of the backward: fp32 dq accumulator (rows x d) + two padded vectors */
  st = attn_bwd_workspace_size(2, 3, 300, 128, &bytes);
  printf("ws %d %lu\n", st, (unsigned long)bytes);
  /* a null q is refused with ATTN_ERR_INVALID_ARG and a message */
  st = attn_fwd(NULL, (void*)0x10000, (void*)0x10000, (void*)0x10000, (float*)0x10000, 1, 1, 128, 64, 0.125f, 0,
                ATTN_BF16, NULL);
  printf("null %d %s|%s\n", st, attn_status_string(st), attn_last_error());
  /* an unsupported head dimension */
  st = attn_fwd((void*)0x10000, (void*)0x10000, (void*)0x10000, (void*)0x10000, (float*)0x10000, 1, 1, 128, 96,
                0.125f, 0, ATTN_BF16, NULL);
  printf("d96 %d\n", st);
  return 0;
}
"""


@pytest.fixture(scope="module")
def gcc():
    path = shutil.which("gcc")
    if path is None:
        pytest.skip("gcc not available")
    return path


@pytest.mark.parametrize("std", ["c89", "c99"])
def test_header_is_plain_c(gcc, tmp_path, std):
    src = tmp_path / "h.c"
    src.write_text('#include "attn_fa2.h"\nint main(void) { return ATTN_OK; }\n')
    r = subprocess.run([gcc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-fsyntax-only", str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_gets_host_side_statuses(gcc, tmp_path, built_library):
    lib_dir = os.path.dirname(built_library)
    src = tmp_path / "caller.c"
    exe = tmp_path / "caller"
    src.write_text(PROGRAM)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", lib_dir, "-lattn_fa2", f"-Wl,-rpath,{lib_dir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = dict(ln.split(" ", 1) for ln in out.stdout.strip().splitlines())
    rows, prows = 2 * 3 * 300, 2 * 3 * 384
    want = -(-rows * 128 * 4 // 256) * 256 + 2 * (-(-prows * 4 // 256) * 256)
    assert lines["ws"] == f"0 {want}"
    st, msg = lines["null"].split(" ", 1)
    assert st == "1" and msg.startswith("invalid argument|") and "null" in msg
    assert lines["d96"] == "2"
