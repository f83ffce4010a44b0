"""The boundary from plain C: a C99 program that includes include/attnfuse.h (no C++, no CUDA
headers), links libattnfuse.so and calls the host-only entry points (version, status strings,
workspace sizes, the mode rule, argument validation).  Runs without a GPU."""
import os
import shutil
import subprocess

import pytest

from attention_rope_causal_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "attnfuse.h"

int main(void) {
  /* host-only calls: no device is touched */
  if (attnfuse_version() == NULL || strlen(attnfuse_version()) == 0) return 1;
  if (strlen(attnfuse_status_string(ATTNFUSE_ERR_INVALID_ARG)) == 0) return 2;
  /* pre-rotate workspace: rotated Q and K, each rounded up to 256 bytes */
  size_t ws = attnfuse_workspace_bytes(1, 32, 8, 4096, 128, ATTNFUSE_PREROTATE, ATTNFUSE_BF16);
  if (ws != (size_t)1 * 4096 * 32 * 128 * 2 + (size_t)1 * 4096 * 8 * 128 * 2) return 3;
  if (attnfuse_workspace_bytes(1, 32, 8, 4096, 128, ATTNFUSE_FUSED, ATTNFUSE_BF16) != 0) return 4;
  /* the measured rule: grouped-query attention from N = 2048 takes the split mode */
  if (attnfuse_select_mode(1, 32, 8, 4096, 128, ATTNFUSE_BF16) != ATTNFUSE_SPLIT) return 5;
  /* arguments are checked before any device work: a null q is refused */
  attnfuse_status_t st = attnfuse_rope_causal_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 2, 128, 64, 1e4,
                                                  ATTNFUSE_FUSED, ATTNFUSE_BF16, NULL, 0, NULL);
  if (st != ATTNFUSE_ERR_INVALID_ARG) return 6;
  printf("ok %s\n", attnfuse_version());
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_program_uses_the_boundary(tmp_path):
    lib = build.build()
    src = tmp_path / "consumer.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", libdir, "-lattnfuse", f"-Wl,-rpath,{libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.startswith("ok ")
