"""The boundary is a plain C ABI: include/thd_attn.h compiles as pedantic C99
(no C++ and no torch types), every function it declares links against the
built library, and a C caller gets the host-side answers without a GPU
(version, status strings, workspace sizes, argument rejections)."""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "thd_attn.h")
LIBDIR = os.path.join(ROOT, "packed_sequence_context_gb300")

C_MAIN = r"""
#include <stdio.h>
#include <string.h>
#include "thd_attn.h"

typedef void (*any_fn)(void);

int main(void) {
  /* every declared entry point, by address: the link fails if one is missing */
  any_fn fns[] = {%s};
  int bad = 0;
  for (size_t i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i) bad |= fns[i] == NULL;
  if (bad) return 10;
  if (thd_version() < 100) return 11;
  if (strcmp(thd_status_string(THD_OK), "ok") != 0) return 12;
  if (strcmp(thd_status_string(9999), "unknown status") != 0) return 13;
  /* workspace sizes: positive for supported sizes, 0 otherwise */
  if (thd_workspace_size(8, 14632, 14632, 16, 16, 128, 4, 1) == 0) return 14;
  if (thd_workspace_size(8, 14632, 14632, 16, 16, 96, 4, 0) != 0) return 15;
  if (thd_a2a_workspace_size(8, 14632, 16, 16, 128, 4, 2, 0) == 0) return 16;
  /* rejected on the host, before any CUDA call */
  if (thd_attn_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 2, 192, 192, 2, 2, 64, 1, 0.125f, 2, -1,
                   NULL, 0, NULL, NULL) != THD_ERR_INVALID_ARG) return 17;
  if (thd_cp_a2a(NULL, NULL, NULL, 2, 192, 4, 64, 4, 2, THD_A2A_TO_GROUPS, NULL, NULL) != THD_ERR_INVALID_ARG)
    return 18;
  if (thd_grad_tail_zero(NULL, NULL, NULL, 192, 192, 2, 2, 64, NULL, NULL, 2, 1, NULL) != THD_OK) return 19;
  printf("c-abi ok\n");
  return 0;
}
"""


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^THD_API\s+[\w\s\*]+?\b(thd_\w+)\s*\(", src, flags=re.M)


def test_header_is_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = os.path.join(LIBDIR, "libthdattn.so")
    if not os.path.exists(lib):
        pytest.skip("library not built")
    names = _declared()
    assert len(names) >= 15
    src = tmp_path / "main.c"
    src.write_text(C_MAIN % ", ".join(f"(any_fn){n}" for n in names))
    exe = tmp_path / "main"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", LIBDIR, "-lthdattn", f"-Wl,-rpath,{LIBDIR}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c-abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
