"""The tensor-core dense pass's operand layouts (tc.cuh, no GPU needed).

The dense pass's MMA descriptors assume 8-row x 16-byte core matrices with
fixed strides (weights: 2048 bytes between K groups, 128 bytes between 8-row
groups; activations: N * 16 and 128), its producer assumes a K chunk of a
tile is one contiguous run, and its tensor-map path assumes that a box of
8 K elements x N rows of a row-major matrix lands exactly as one K group of
the activation layout.  This compiles the layout functions on the host (nvcc)
and checks each of those properties, plus that both layouts are bijections
onto their byte ranges."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_decode_step_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "tc.cuh"
using namespace moe;

static int fails = 0;
#define CHECK(c, what) do { if (!(c)) { ++fails; std::printf("FAIL %s\n", what); return; } } while (0)

static void weights(int K, int KC) {
  const size_t tile = (size_t)256 * K;
  std::vector<int> seen(tile / 2, 0);
  for (int T = 0; T < 2; ++T)
    for (int m = 0; m < 128; ++m)
      for (int k = 0; k < K; ++k) {
        const size_t o = dense_w_offset(K, T, m, k);
        CHECK(o % 2 == 0 && o >= (size_t)T * tile && o < (size_t)(T + 1) * tile, "weight offset range");
        if (T == 0) seen[o / 2]++;
        if (k % 8 == 0 && k + 8 < K)
          CHECK(dense_w_offset(K, T, m, k + 8) - o == 2048, "weight LBO (K groups 2048 B apart)");
        if (m % 8 == 0 && m + 8 < 128)
          CHECK(dense_w_offset(K, T, m + 8, k) - o == 128, "weight SBO (row groups 128 B apart)");
        if (m % 8 != 7) CHECK(dense_w_offset(K, T, m + 1, k) - o == 16, "core matrix rows 16 B apart");
        if (k % 8 != 7) CHECK(dense_w_offset(K, T, m, k + 1) - o == 2, "core matrix row contiguous");
        if (k + 16 < K) CHECK(dense_w_offset(K, T, m, k + 16) - o == 4096, "MMA K step of 4 KB");
        const size_t c = (size_t)(k / KC);
        CHECK(o - (size_t)T * tile >= c * 256 * KC && o - (size_t)T * tile < (c + 1) * 256 * KC,
              "a K chunk of a tile is one contiguous run");
      }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "weight layout is a bijection");
}

static void activations(int NP, int K, int KC) {
  std::vector<int> seen((size_t)NP * K, 0);
  for (int n = 0; n < NP; ++n)
    for (int k = 0; k < K; ++k) {
      const size_t o = dense_act_offset(NP, n, k);
      CHECK(o % 2 == 0 && o < (size_t)NP * K * 2, "activation offset range");
      seen[o / 2]++;
      if (k % 8 == 0 && k + 8 < K)
        CHECK(dense_act_offset(NP, n, k + 8) - o == (size_t)NP * 16, "activation LBO (N * 16 B)");
      if (n % 8 == 0 && n + 8 < NP) CHECK(dense_act_offset(NP, n + 8, k) - o == 128, "activation SBO");
      if (k + 16 < K)
        CHECK(dense_act_offset(NP, n, k + 16) - o == (size_t)32 * NP, "activation MMA K step");
      const size_t c = (size_t)(k / KC);
      CHECK(o >= c * NP * KC * 2 && o < (c + 1) * NP * KC * 2, "an activation chunk is contiguous");
      // a tensor-map box of 8 K elements x NP rows at (8 g, 0) writes element
      // (n, 8 g + j) at n * 16 + 2 j of its destination, g * NP * 16 into the chunk
      const size_t box = (size_t)(k / 8) * NP * 16 + (size_t)n * 16 + (size_t)(k % 8) * 2;
      CHECK(box == o, "tensor-map box order equals the activation layout");
    }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "activation layout is a bijection");
}

int main() {
  weights(256, 128);
  weights(512, 64);
  for (int NP : {16, 48, 64, 128}) activations(NP, 256, NP <= 64 ? 128 : 64);
  CHECK(dense_np(1) == 16 && dense_np(16) == 16 && dense_np(17) == 32 && dense_np(128) == 128, "dense_np");
  CHECK(dense_stage_bytes(128, 64) == 49152 && dense_stage_bytes(64, 128) == 32768, "stage bytes");
  std::printf("%s %d\n", fails ? "FAILED" : "PASSED", fails);
  return fails ? 1 : 0;
}
"""


def test_dense_operand_layouts(tmp_path):
    nvcc = shutil.which("nvcc") or (os.path.exists("/usr/local/cuda/bin/nvcc")
                                    and "/usr/local/cuda/bin/nvcc")
    if not nvcc:
        pytest.skip("nvcc not available")
    src = tmp_path / "dense_layout.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "dense_layout"
    subprocess.check_call([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                           str(src)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and "PASSED 0" in out.stdout, out.stdout + out.stderr
