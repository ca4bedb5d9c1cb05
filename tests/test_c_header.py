"""include/specverify.h is a C header: a C11 program that includes it builds
with warnings as errors, links against libspecverify.so and calls the
host-side entry points (sizes, version, host-checked errors).  None of these
calls reaches a device, so this runs without a GPU."""

import os
import shutil
import subprocess

import pytest

from speculative_decoding_verification_47_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "specverify.h"

int main(void) {
  int32_t dummy[4];
  sv_status s;
  if (sv_version() < 100) return 1;
  if (sv_workspace_size(256, 8, 128256, SV_BF16) == 0) return 2;
  if (sv_workspace_size(0, 8, 128256, SV_BF16) != 0) return 3;
  if (sv_draft_sample_workspace_size() < 4) return 4;
  if (sv_dynk_state_size(256) < 256 * 156) return 5;
  if (sv_lmhead_workspace_size(512, 4096) == 0) return 6;
  /* B = 0: rejected on the host, before any device work */
  s = sv_spec_verify(dummy, 0, 0, dummy, 0, 0, SV_BF16, 0, 3, 100, dummy, NULL, NULL, 1.0f,
                     (const float*)dummy, NULL, dummy, dummy, NULL, dummy, 1024, NULL);
  if (s != SV_ERR_SHAPE || strlen(sv_last_error()) == 0) return 7;
  s = sv_kv_commit(NULL, dummy, NULL, NULL, 4, 3, dummy, 256, NULL);
  if (s != SV_ERR_ARG) return 8;
  printf("ok %d\n", sv_version());
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_and_links_as_c(tmp_path):
    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
           f"-L{libdir}", "-l:libspecverify.so", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr)
