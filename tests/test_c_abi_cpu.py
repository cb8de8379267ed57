"""The C ABI from C: include/gva.h compiles as strict C99, a C program links libgva.so and
calls the entry points that need no GPU (version, status strings, host-side rejection)."""
import os
import shutil
import subprocess

import pytest

from compact_kv_cache_gva_b300 import gva

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gva.h"

int main(void) {
  gva_dims d = {16, 4, 64, 64, 16, GVA_BLOCK_TOKENS, GVA_BF16, 10000.0, 0.0f};
  gva_ctx* ctx = NULL;
  if (gva_version() < 100) return 1;
  if (strcmp(gva_status_string(GVA_OK), "ok") != 0) return 2;
  /* null contexts are rejected on the host, before any CUDA call */
  if (gva_decode_step(NULL, 1, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, NULL, 1, NULL, NULL, 0,
                      NULL) != GVA_ERR_INVALID_ARG)
    return 3;
  if (gva_decode_attention(NULL, 1, NULL, NULL, NULL, NULL, NULL, 1, 1, NULL, 1, NULL, NULL, 0, NULL) !=
      GVA_ERR_INVALID_ARG)
    return 4;
  if (gva_decode_step_workspace_size(NULL, 1, 1) != 0 || gva_step_is_fused(NULL, 1, 1) != -1) return 5;
  /* bad dims are rejected before the context touches the device */
  d.H = 6;
  if (gva_create(&d, &ctx) != GVA_ERR_INVALID_ARG || ctx != NULL) return 6;
  printf("ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_the_library_links_from_c(tmp_path):
    if not os.path.exists(gva.LIB_PATH):
        from compact_kv_cache_gva_b300 import build
        build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(gva.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lgva", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.strip() == "ok"
