"""The header is plain C: a C99 program that includes include/moe.h, links
against libmoe_b300.so and calls the host-only entry points (shape checks,
workspace and capacity sizes, error strings) builds with gcc and runs on a
machine without a GPU."""
import os
import shutil
import subprocess

import pytest

from top_routing_expert_lb_b300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include "moe.h"

int main(void) {
  moe_shape_t s = {4096, 4096, 14336, 8, 2, 0, 1.25f, 0.01f, 0u};
  size_t ws = 0;
  int64_t C = 0, rows = 0;
  if (moe_workspace_size(&s, &ws) != MOE_OK || ws == 0) return 1;
  if (moe_capacity(&s, &C) != MOE_OK) return 2;
  if (moe_max_rows(&s, &rows) != MOE_OK) return 3;
  s.k = 9;  /* k > E: refused */
  if (moe_workspace_size(&s, &ws) != MOE_ERR_INVALID_ARG) return 4;
  s.k = 2;
  s.tuning.gemm1_tile = 64;  /* not a tile height the library has: refused */
  if (moe_workspace_size(&s, &ws) != MOE_ERR_INVALID_ARG) return 5;
  s.tuning.gemm1_tile = 256;  /* CTA-pair gate/up tiles: accepted */
  s.tuning.options = MOE_TUNE_NO_HALF_TILES;
  if (moe_workspace_size(&s, &ws) != MOE_OK) return 6;
  printf("C=%lld rows=%lld err=%s\n", (long long)C, (long long)rows,
         moe_error_string(MOE_ERR_TIMEOUT));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_builds_and_runs(tmp_path):
    lib = mbuild.ensure_built()
    libdir = os.path.dirname(lib)
    src = tmp_path / "client.c"
    src.write_text(C_SRC)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-lmoe_b300", "-Wl,-rpath," + libdir, "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    # C = ceil(1.25 * 2 * 4096 / 8) = 1280 per expert; rows = min(T k, E C) = 8192
    assert out.startswith("C=1280 rows=8192 err=")
