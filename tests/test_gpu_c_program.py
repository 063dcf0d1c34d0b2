"""The device path driven from C with raw device pointers (no torch): a C99
program allocates with cudaMalloc, calls reshape_and_cache and
paged_attention_decode through include/pagedkv.h, and writes the cache and the
output back.  The tiny fp32 workload's inputs come from the oracle pool; the
cache bytes must equal the oracle's append and the output its attention."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import workloads as W
from tests import gpu_cases as GC

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "paged_kv_cache_295_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "pagedkv.h"

static void* load(FILE* f, size_t n) {
  void* p = malloc(n);
  if (!p || fread(p, 1, n, f) != n) { fprintf(stderr, "short input\n"); exit(2); }
  return p;
}
static void* to_dev(const void* h, size_t n) {
  void* d = NULL;
  if (cudaMalloc(&d, n) != cudaSuccess || cudaMemcpy(d, h, n, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "cuda\n"); exit(3);
  }
  return d;
}

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 1;
  int32_t hdr[8];  /* S, Hq, Hkv, D, bs, NB, MB, max_ctx */
  if (fread(hdr, 4, 8, f) != 8) return 1;
  const int32_t S = hdr[0], Hq = hdr[1], Hkv = hdr[2], D = hdr[3], bs = hdr[4], NB = hdr[5],
                MB = hdr[6], max_ctx = hdr[7];
  const size_t cache_n = (size_t)NB * bs * Hkv * D * 4;
  float* q = load(f, (size_t)S * Hq * D * 4);
  float* kc = load(f, cache_n);
  float* vc = load(f, cache_n);
  int32_t* bt = load(f, (size_t)S * MB * 4);
  int32_t* cl = load(f, (size_t)S * 4);
  float* kn = load(f, (size_t)S * Hkv * D * 4);
  float* vn = load(f, (size_t)S * Hkv * D * 4);
  int64_t* sl = load(f, (size_t)S * 8);
  fclose(f);

  void* d_q = to_dev(q, (size_t)S * Hq * D * 4);
  void* d_kc = to_dev(kc, cache_n);
  void* d_vc = to_dev(vc, cache_n);
  int32_t* d_bt = to_dev(bt, (size_t)S * MB * 4);
  int32_t* d_cl = to_dev(cl, (size_t)S * 4);
  void* d_kn = to_dev(kn, (size_t)S * Hkv * D * 4);
  void* d_vn = to_dev(vn, (size_t)S * Hkv * D * 4);
  int64_t* d_sl = to_dev(sl, (size_t)S * 8);
  int32_t zero = 0;
  int32_t* d_status = to_dev(&zero, 4);
  float* d_out = NULL;
  if (cudaMalloc((void**)&d_out, (size_t)S * Hq * D * 4) != cudaSuccess) return 3;
  const size_t ws_n = paged_attention_workspace_bytes(S, Hq, Hkv, D, max_ctx, 0);
  void* d_ws = NULL;
  if (ws_n && cudaMalloc(&d_ws, ws_n) != cudaSuccess) return 3;

  pkv_status st = reshape_and_cache(d_kn, d_vn, d_sl, d_kc, d_vc, S, Hkv, D, bs, NB, PKV_F32,
                                    PKV_F32, NULL, NULL, d_status, NULL);
  if (st != PKV_OK) { fprintf(stderr, "append %d\n", (int)st); return 4; }
  st = paged_attention_decode(d_q, d_kc, d_vc, d_bt, d_cl, S, Hq, Hkv, D, bs, NB, MB, max_ctx,
                              0.125f, PKV_F32, PKV_F32, NULL, NULL, d_out, d_ws, ws_n, 0, d_status,
                              NULL);
  if (st != PKV_OK) { fprintf(stderr, "decode %d\n", (int)st); return 5; }
  if (cudaDeviceSynchronize() != cudaSuccess) return 6;

  float* out = malloc((size_t)S * Hq * D * 4);
  int32_t status = -1;
  cudaMemcpy(out, d_out, (size_t)S * Hq * D * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(kc, d_kc, cache_n, cudaMemcpyDeviceToHost);
  cudaMemcpy(vc, d_vc, cache_n, cudaMemcpyDeviceToHost);
  cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost);
  FILE* g = fopen(argv[2], "wb");
  if (!g) return 7;
  fwrite(&status, 4, 1, g);
  fwrite(out, 4, (size_t)S * Hq * D, g);
  fwrite(kc, 1, cache_n, g);
  fwrite(vc, 1, cache_n, g);
  fclose(g);
  return 0;
}
"""


def test_decode_step_from_a_c_program(lib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "step.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "step"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), str(src), "-o", str(exe),
                    "-L", LIB_DIR, "-lpagedkv", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + LIB_DIR + ":" + os.path.join(CUDA, "lib64")], check=True)

    w = W.TINY
    assert abs(w.scale - 0.125) < 1e-12                # the program passes 1/sqrt(64)
    case, _ = GC.make_small(w)
    kc0, vc0 = GC.oracle_caches(case, 0)            # after prompts and the step's append
    nb, bs, hkv, d = case.nb, w.block_size, w.num_kv_heads, w.head_dim
    # the program appends the step itself: start from the cache before that append
    kc_in = np.full((nb, bs, hkv, d), np.nan, dtype=np.float32)
    vc_in = np.full((nb, bs, hkv, d), np.nan, dtype=np.float32)
    from oracle import attention as OA
    OA.reshape_and_cache(case.prompt_k[0], case.prompt_v[0], case.prompt_slots, kc_in, vc_in,
                         "f32", "f32")
    S, mb = len(case.lens), case.tables.shape[1]
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        np.array([S, w.num_q_heads, hkv, d, bs, nb, mb, int(case.lens.max())],
                 dtype=np.int32).tofile(f)
        for a, dt in ((case.q[0], np.float32), (kc_in, np.float32), (vc_in, np.float32),
                      (case.tables, np.int32), (case.lens, np.int32),
                      (case.k_new[0], np.float32), (case.v_new[0], np.float32),
                      (case.step_slots, np.int64)):
            np.ascontiguousarray(a, dtype=dt).tofile(f)
    res = tmp_path / "out.bin"
    subprocess.run([str(exe), str(inp), str(res)], check=True)
    raw = np.fromfile(res, dtype=np.uint8)
    status = int(raw[:4].view(np.int32)[0])
    n_out = S * w.num_q_heads * d * 4
    out = raw[4:4 + n_out].view(np.float32).reshape(S, w.num_q_heads, d)
    cn = nb * bs * hkv * d * 4
    kc = raw[4 + n_out:4 + n_out + cn].view(np.float32).reshape(kc0.shape)
    vc = raw[4 + n_out + cn:4 + n_out + 2 * cn].view(np.float32).reshape(vc0.shape)
    assert status == 0
    assert kc.tobytes() == kc0.astype(np.float32).tobytes()
    assert vc.tobytes() == vc0.astype(np.float32).tobytes()
    ref = GC.oracle_out(case, 0, kc0, vc0)
    assert np.abs(out.astype(np.float64) - ref).max() <= 2e-3
