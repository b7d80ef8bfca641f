"""The C ABI used from plain C (no Python between the caller and libsfa.so):
small C programs written here are compiled with gcc against include/sfa.h
and linked with the in-tree libsfa.so.  The host program runs anywhere; the
device program (marked gpu) runs a forward through the C calls alone."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "static_offset_sparse_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")

HOST_C = r"""
#include <stdio.h>
#include <stdint.h>
#include "sfa.h"

int main(void) {
  int32_t fib[15], ch[200], n = 0, delta = 0, starts[8], lens[8], nruns = 0;
  if (sfa_offsets_fib(15, fib) != SFA_OK) return 1;
  if (sfa_offsets_christoffel(128, 1024, 1, ch, 200, &n) != SFA_OK) return 2;
  if (sfa_band_plan(ch, n, 2048, 1, &delta, starts, lens, 8, &nruns) != SFA_OK) return 3;
  printf("fib");
  for (int i = 0; i < 15; ++i) printf(" %d", fib[i]);
  printf("\nchristoffel %d %d %d %d\n", n, ch[0], ch[1], ch[n - 1]);
  printf("band %d %d", delta, nruns);
  for (int m = 0; m < nruns; ++m) printf(" %d:%d", starts[m], lens[m]);
  printf("\nstatus %s\n", sfa_status_string(SFA_ERR_CAPACITY));
  return 0;
}
"""

DEVICE_C = r"""
#include <stdio.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "sfa.h"

static uint16_t to_bf16(float f) { uint32_t u; memcpy(&u, &f, 4); return (uint16_t)(u >> 16); }

static void fill(uint16_t* h, size_t n, uint32_t* state) {
  for (size_t i = 0; i < n; ++i) {
    *state = *state * 1664525u + 1013904223u;
    h[i] = to_bf16(((float)(*state >> 8) / 16777216.0f) * 2.0f - 1.0f);
  }
}

#define CK(x) do { if ((x) != cudaSuccess) { printf("cuda error line %d\n", __LINE__); return 10; } } while (0)

int main(void) {
  const int B = 2, T = 100, Hq = 8, Hkv = 2, D = 64, G = Hq / Hkv;
  const size_t nq = (size_t)B * Hq * T * D, nk = (size_t)B * Hkv * T * D;
  uint16_t* hq = malloc(nq * 2); uint16_t* hk = malloc(nk * 2);
  uint16_t* hv = malloc(nk * 2); uint16_t* ho = malloc(nq * 2);
  uint32_t st = 12345u;
  fill(hq, nq, &st); fill(hk, nk, &st); fill(hv, nk, &st);
  void *q, *k, *v, *o; float *lse, *rope; size_t rope_bytes = 0;
  CK(cudaMalloc(&q, nq * 2)); CK(cudaMalloc(&k, nk * 2)); CK(cudaMalloc(&v, nk * 2));
  CK(cudaMalloc(&o, nq * 2)); CK(cudaMalloc((void**)&lse, (size_t)B * Hq * T * 4));
  if (sfa_rope_table_bytes(T, &rope_bytes) != SFA_OK) return 2;
  CK(cudaMalloc((void**)&rope, rope_bytes));
  CK(cudaMemcpy(q, hq, nq * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(k, hk, nk * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(v, hv, nk * 2, cudaMemcpyHostToDevice));
  if (sfa_rope_table(T, 1e4, rope, NULL) != SFA_OK) return 3;
  /* keys: distance 0 only, so each query's softmax has one key and O = V exactly */
  int32_t dist[1] = {0};
  sfa_desc d;
  memset(&d, 0, sizeof d);
  d.B = B; d.T = T; d.Hq = Hq; d.Hkv = Hkv; d.D = D; d.dtype = SFA_BF16;
  d.dist = dist; d.n_dist = 1; d.rope = rope;
  size_t ws_bytes = 0; void* ws = NULL;
  if (sfa_workspace_size(&d, 0, 0, &ws_bytes) != SFA_OK) return 4;
  if (ws_bytes) CK(cudaMalloc(&ws, ws_bytes));
  int rc = sfa_forward_int(&d, q, k, v, o, lse, ws, ws_bytes, NULL);
  if (rc != SFA_OK) { printf("forward rc %d %s\n", rc, sfa_status_string(rc)); return 5; }
  CK(cudaDeviceSynchronize());
  int32_t status = -1;
  if (sfa_get_device_status(NULL, &status) != SFA_OK || status != 0) return 6;
  CK(cudaMemcpy(ho, o, nq * 2, cudaMemcpyDeviceToHost));
  size_t bad = 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h)
      for (int t = 0; t < T; ++t)
        for (int e = 0; e < D; ++e) {
          size_t io = (((size_t)b * Hq + h) * T + t) * D + e;
          size_t iv = (((size_t)b * Hkv + h / G) * T + t) * D + e;
          bad += ho[io] != hv[iv];
        }
  printf("mismatches %zu of %zu\n", bad, nq);
  return bad ? 7 : 0;
}
"""


def _build(tmp_path, src, name, cflags=(), libs=()):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not available")
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    exe = tmp_path / name
    cmd = [gcc, "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"), *cflags, str(c), "-L", PKG,
           "-lsfa", f"-Wl,-rpath,{PKG}", *libs, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe):
    env = dict(os.environ, LD_LIBRARY_PATH=PKG + os.pathsep + os.environ.get("LD_LIBRARY_PATH", ""))
    return subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)


def test_host_calls_from_c(sfa_lib, tmp_path):
    exe = _build(tmp_path, HOST_C, "host_calls")
    r = _run(exe)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    lines = r.stdout.splitlines()
    assert lines[0] == "fib 1 2 3 5 8 13 21 34 55 89 144 233 377 610 987"
    assert lines[1] == "christoffel 129 0 7 1023"
    assert lines[2] == "band 8 2 0:1 7:128"
    assert lines[3].startswith("status ")


@pytest.mark.gpu
def test_device_forward_from_c(sfa_lib, tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib64 = os.path.join(CUDA, "lib64")
    exe = _build(tmp_path, DEVICE_C, "device_forward", cflags=["-I", os.path.join(CUDA, "include")],
                 libs=["-L", lib64, "-lcudart", f"-Wl,-rpath,{lib64}"])
    r = _run(exe)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "mismatches 0 of" in r.stdout
