"""The boundary from plain C: a C99 program that includes include/mla.h,
links libmla.so and calls its host-side entry points (CPU only).

It checks that the header compiles as C with warnings as errors, that the
library links from C, that the host planner run from C writes the same
metadata as through the Python binding, and that a launching call with bad
arguments returns MLA_ERR_INVALID_ARG instead of reaching a GPU."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from mla_decode_attention_07_gb300 import libmla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include "mla.h"

int main(int argc, char** argv) {
  if (argc != 2) return 2;
  const int32_t lens[3] = {130, 0, 4096};
  const int clusters = 76;
  size_t bytes = mla_plan_size_for_clusters(3, 2, 16, clusters);
  if (bytes == 0) return 3;
  void* plan = calloc(1, bytes);
  if (!plan) return 4;
  int rc = mla_decode_plan_host(lens, 3, 2, 16, clusters, plan, bytes);
  if (rc != MLA_OK) return 5;
  FILE* f = fopen(argv[1], "wb");
  if (!f || fwrite(plan, 1, bytes, f) != bytes) return 6;
  fclose(f);
  /* a launching call with a null query is rejected on the host */
  rc = mla_decode(NULL, NULL, 0, NULL, 0, NULL, 3, 2, 16, plan, NULL, NULL, 0.1f, NULL, 0, NULL);
  if (rc != MLA_ERR_INVALID_ARG) return 7;
  if (mla_strerror(rc) == NULL || strlen(mla_strerror(rc)) == 0) return 8;
  if (mla_decode_plan_host(lens, 3, 2, 16, clusters, plan, 8) != MLA_ERR_WORKSPACE) return 9;
  free(plan);
  printf("ok %zu\n", bytes);
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    import __graft_entry__
    return __graft_entry__.build_library()


def test_c_program_uses_the_abi(lib_path, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    lib_dir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", str(src), "-I", os.path.join(ROOT, "include"),
           "-o", str(exe), lib_path, f"-Wl,-rpath,{lib_dir}"]
    built = subprocess.run(cmd, capture_output=True, text=True)
    assert built.returncode == 0, built.stderr
    out_file = tmp_path / "plan.bin"
    run = subprocess.run([str(exe), str(out_file)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    from_c = np.fromfile(out_file, dtype=np.int32)
    from_py = libmla.mla_decode_plan_host(np.array([130, 0, 4096], dtype=np.int32), 2, 16, 76)
    assert np.array_equal(from_c, np.asarray(from_py).view(np.int32).ravel()[: from_c.size])
