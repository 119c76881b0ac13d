"""The boundary from plain C: C99 programs that include include/mla.h and
link libmla.so, with no Python or PyTorch in the process.

On the CPU: the header compiles as C with warnings as errors, the library
links from C, the host planner run from C writes the same metadata as
through the Python binding, and a launching call with bad arguments returns
MLA_ERR_INVALID_ARG instead of reaching a GPU.  On a GB300 (marked gpu): a C
program allocates device memory with the CUDA runtime, plans and decodes a
small ragged batch (one entry empty) through the C ABI, and its out and lse
match the fp64 oracle within the fixed tolerances."""
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


GPU_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime_api.h>
#include "mla.h"

static void* slurp(const char* dir, const char* name, size_t* n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  *n = (size_t)ftell(f);
  fseek(f, 0, SEEK_SET);
  void* p = malloc(*n ? *n : 1);
  if (p && fread(p, 1, *n, f) != *n) { free(p); p = NULL; }
  fclose(f);
  return p;
}

static void* to_device(const void* h, size_t n) {
  void* d = NULL;
  if (cudaMalloc(&d, n ? n : 16) != cudaSuccess) return NULL;
  if (n && cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

static int spill(const char* dir, const char* name, const void* d, size_t n) {
  char path[4096];
  void* h = malloc(n);
  if (!h || cudaMemcpy(h, d, n, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(h, 1, n, f) != n) return 1;
  fclose(f);
  free(h);
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 8) return 2;
  const char* dir = argv[1];
  const int batch = atoi(argv[2]), s_q = atoi(argv[3]), h_q = atoi(argv[4]);
  const int num_pages = atoi(argv[5]), max_pages = atoi(argv[6]);
  const float scale = (float)atof(argv[7]);
  size_t nq, nkv, nbt, nsl;
  void* hq = slurp(dir, "q.bin", &nq);
  void* hkv = slurp(dir, "kv.bin", &nkv);
  void* hbt = slurp(dir, "bt.bin", &nbt);
  void* hsl = slurp(dir, "sl.bin", &nsl);
  if (!hq || !hkv || !hbt || !hsl) return 3;
  void* q = to_device(hq, nq);
  void* kv = to_device(hkv, nkv);
  void* bt = to_device(hbt, nbt);
  void* sl = to_device(hsl, nsl);
  const size_t rows = (size_t)batch * s_q * h_q;
  const size_t plan_bytes = mla_plan_size(batch, s_q, h_q, 0);
  const size_t ws_bytes = mla_workspace_size(batch, s_q, h_q, 0);
  if (!plan_bytes || !ws_bytes) return 4;
  void *plan = NULL, *ws = NULL, *out = NULL, *lse = NULL;
  if (cudaMalloc(&plan, plan_bytes) || cudaMalloc(&ws, ws_bytes) ||
      cudaMalloc(&out, rows * 512 * 2) || cudaMalloc(&lse, rows * 4))
    return 5;
  if (!q || !kv || !bt || !sl) return 6;
  int rc = mla_decode_plan((const int32_t*)sl, batch, s_q, h_q, plan, plan_bytes, NULL);
  if (rc != MLA_OK) { fprintf(stderr, "plan: %s\n", mla_strerror(rc)); return 7; }
  rc = mla_decode(q, kv, num_pages, (const int32_t*)bt, max_pages, (const int32_t*)sl, batch,
                  s_q, h_q, plan, out, (float*)lse, scale, ws, ws_bytes, NULL);
  if (rc != MLA_OK) { fprintf(stderr, "decode: %s\n", mla_strerror(rc)); return 8; }
  rc = mla_check_device_error(NULL);
  if (rc != MLA_OK) { fprintf(stderr, "device: %s\n", mla_strerror(rc)); return 9; }
  if (spill(dir, "out.bin", out, rows * 512 * 2) || spill(dir, "lse.bin", lse, rows * 4)) return 10;
  printf("ok\n");
  return 0;
}
"""


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    return None


@pytest.mark.gpu
def test_c_program_decodes_on_the_gpu(lib_path, tmp_path, oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = _cuda_home()
    if cc is None or cuda is None:
        pytest.skip("no C compiler or CUDA headers")
    from mla_decode_attention_07_gb300 import workloads as W
    inp = W.make_inputs(seed=61, batch=3, s_q=2, h_q=16, seqlens=[700, 0, 130], extra_pages=2)
    np.ascontiguousarray(inp.q).tofile(tmp_path / "q.bin")
    np.ascontiguousarray(inp.kv_cache).tofile(tmp_path / "kv.bin")
    np.ascontiguousarray(inp.block_table, dtype=np.int32).tofile(tmp_path / "bt.bin")
    np.ascontiguousarray(inp.cache_seqlens, dtype=np.int32).tofile(tmp_path / "sl.bin")
    src = tmp_path / "gpu_client.c"
    src.write_text(GPU_SOURCE)
    exe = tmp_path / "gpu_client"
    lib_dir = os.path.dirname(lib_path)
    cmd = [cc, "-std=c99", "-Wall", "-Werror", str(src), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-o", str(exe), lib_path,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", f"-Wl,-rpath,{lib_dir}",
           f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    built = subprocess.run(cmd, capture_output=True, text=True)
    assert built.returncode == 0, built.stderr
    B, s_q, h_q = inp.batch, inp.s_q, inp.h_q
    run = subprocess.run([str(exe), str(tmp_path), str(B), str(s_q), str(h_q),
                          str(inp.kv_cache.shape[0]), str(inp.block_table.shape[1]),
                          repr(float(inp.softmax_scale))],
                         capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    out = W.bf16_bits_to_float32(np.fromfile(tmp_path / "out.bin", dtype=np.uint16))
    out = out.reshape(B, s_q, h_q, 512).astype(np.float64)
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32).reshape(B, h_q, s_q).astype(np.float64)
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    empty = np.isneginf(ref_l)
    assert empty[1].all() and not empty[0].any()
    assert np.array_equal(np.isneginf(lse), empty)
    assert float(np.abs(out - ref_o).max()) <= 1e-2
    assert float(np.abs(np.where(empty, 0.0, lse) - np.where(empty, 0.0, ref_l)).max()) <= 1e-3
