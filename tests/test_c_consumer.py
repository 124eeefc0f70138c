"""The boundary is a C ABI: a plain C11 program (no C++, -pedantic, warnings as errors)
includes include/mla.h, links the shared library and calls its host-only entry points.
No GPU is needed: nothing here launches a kernel."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "mla_latent_kv_69_b300", "lib")

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "mla.h"

int main(void) {
  int st = -1, en = -1;
  if (mla_split_range(1000, 3, 1, &st, &en) != MLA_OK) return 1;
  if (mla_split_range(-1, 3, 1, &st, &en) != MLA_ERR_INVALID_ARG) return 2;
  if (mla_decode_kernel(MLA_KV_BF16, 128) != MLA_KERNEL_TC_BF16) return 3;
  if (mla_decode_kernel(MLA_KV_FP8_E4M3, 128) != MLA_KERNEL_TC_E4M3) return 4;
  if (mla_decode_kernel(MLA_KV_BF16, 7) != -1) return 5;
  if (strncmp(mla_status_string(MLA_ERR_TIMEOUT), "MLA_ERR_TIMEOUT", 15) != 0) return 6;
  /* argument checks run on the host, before any CUDA call */
  if (mla_absorb_q(NULL, NULL, NULL, 1, 128, 10000.f, NULL, 0) != MLA_ERR_INVALID_ARG) return 7;
  if (mla_combine(NULL, NULL, 1, 1, 128, NULL, NULL, 0) != MLA_ERR_INVALID_ARG) return 8;
  if (mla_combine_up_v(NULL, NULL, 1, 1, 128, NULL, NULL, NULL, NULL, 0) != MLA_ERR_INVALID_ARG) return 9;
  printf("%d %d %d\n", st, en, mla_abi_version());
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_plain_c_program_builds_against_the_header_and_runs(tmp_path):
    src = tmp_path / "consumer.c"
    exe = tmp_path / "consumer"
    src.write_text(C_SOURCE)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    build = subprocess.run(
        ["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
         "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src),
         "-L", LIB_DIR, "-lmla_b300", f"-Wl,-rpath,{LIB_DIR}", "-o", str(exe)],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, f"check {run.returncode} failed: {run.stdout}{run.stderr}"
    st, en, abi = (int(v) for v in run.stdout.split())
    assert (st, en) == (384, 768) and abi >= 1
