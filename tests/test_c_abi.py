"""The boundary is plain C: a C99 program includes jattn.h with every warning
as an error, links libjattn.so and calls the entry points that need no GPU
(version, status and kernel names, and argument validation, which returns
before any CUDA call)."""
import os
import shutil
import subprocess

import pytest

from joint_attention_gb300.build import INCLUDE, build

C_PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "jattn.h"

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("failed: %s\n", #cond); ++fails; } } while (0)

int main(void) {
  int cu_bad[3] = {0, 5, 3};
  int cu_ok[3] = {0, 5, 9};
  EXPECT(jattn_version() >= 100);
  EXPECT(strcmp(jattn_status_string(JATTN_OK), jattn_status_string(JATTN_ERR_TIMEOUT)) != 0);
  EXPECT(strcmp(jattn_kernel_name(JATTN_KERNEL_ATTN_BWD), "attn_bwd") == 0);
  EXPECT(JATTN_KERNEL_COUNT == 6);
  /* null pointers and bad shapes are rejected before anything is enqueued */
  EXPECT(jattn_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 16, 8, 64, NULL, NULL, NULL) == JATTN_ERR_INVALID_ARG);
  EXPECT(jattn_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                   1, 1, 16, 8, 64, NULL) == JATTN_ERR_INVALID_ARG);
  EXPECT(jattn_fwd_noalloc(NULL, NULL, NULL, NULL, NULL, 1, 1, 16, 8, 64, NULL, NULL, NULL) ==
         JATTN_ERR_INVALID_ARG);
  EXPECT(jattn_fwd_varlen(NULL, NULL, NULL, NULL, NULL, cu_bad, 2, 2, 64, NULL, NULL, NULL) ==
         JATTN_ERR_INVALID_ARG);
  EXPECT(jattn_bwd_varlen(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                          cu_ok, 2, 2, 64, NULL) == JATTN_ERR_INVALID_ARG);
  EXPECT(jattn_profile_read(JATTN_KERNEL_COUNT, NULL, NULL) != JATTN_OK);
  EXPECT(JATTN_MAX_SEQS == 256);
  printf("%s\n", fails ? "FAILED" : "c abi ok");
  return fails;
}
"""


@pytest.fixture(scope="module")
def libpath():
    return build()


def test_c99_program_includes_the_header_links_and_runs(libpath, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(libpath)
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
           "-L", libdir, "-ljattn", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, r.stdout + r.stderr
