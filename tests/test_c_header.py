"""The boundary from C: include/moe.h compiles as plain C11 (no C++ types, no
CUDA headers needed), and a C program linked against the library queries a
workspace size, reads status strings and has an invalid call rejected -- all
on the host, no GPU."""
import os
import shutil
import subprocess

import pytest

from routing_dispatch_expert_05_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  moe_config_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n_tokens = 16384; cfg.d_model = 2048; cfg.n_experts = 128; cfg.top_k = 8;
  cfg.d_ff = 768; cfg.route = MOE_ROUTE_TOPK_SOFTMAX; cfg.expert = MOE_EXPERT_SWIGLU;
  cfg.dtype = MOE_BF16; cfg.balance_coef = 0.01f;
  size_t bytes = 0;
  if (moe_workspace_size(&cfg, &bytes) != MOE_OK || bytes == 0) return 1;
  printf("workspace %zu\n", bytes);
  printf("status %s | %s\n", moe_status_string(MOE_OK),
         moe_status_string(MOE_ERR_WORKSPACE));
  cfg.top_k = 0;                                /* invalid: rejected on the host */
  if (moe_workspace_size(&cfg, &bytes) != MOE_ERR_INVALID_ARG) return 2;
  moe_weights_t w;
  memset(&w, 0, sizeof w);
  cfg.top_k = 8;
  /* no weights, no workspace: refused before anything reaches a device */
  if (moe_forward(&cfg, NULL, &w, NULL, NULL, NULL, 0, NULL) != MOE_ERR_INVALID_ARG) return 3;
  printf("version %d\n", moe_version());
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_as_c_and_the_library_links(tmp_path):
    lib = B.build()
    src = tmp_path / "use_moe.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_moe"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    lines = r.stdout.splitlines()
    assert lines[0].startswith("workspace ") and int(lines[0].split()[1]) > 1 << 30
    assert lines[1] == "status ok | workspace too small"
    assert lines[2].startswith("version ")
