"""Host-side checks of the launch order the kernels share (csrc/internal.h), compiled
with the host C++ compiler (no GPU needed): grouped_tile_head maps the linear grid
position onto every (tile, head) pair exactly once, puts every head's tile 0 (the
longest causal work) first within its group, and keeps groups in order; head_group
sizes groups to about 32 MiB of Q, K, V, dO and stays within [1, B*H]."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_26_gb300", "csrc")

CHECKER = r"""
#include <cstdio>
#include <vector>
#include "internal.h"
int main() {
  const int Ts[] = {1, 2, 3, 7, 32, 64, 256};
  const int BHs[] = {1, 2, 5, 31, 32, 33, 512};
  const int hgs[] = {1, 2, 3, 4, 8, 16, 1000};
  for (int T : Ts) for (int BH : BHs) for (int hg0 : hgs) {
    const int hg = hg0 < BH ? hg0 : BH;
    std::vector<int> seen(static_cast<size_t>(T) * BH, 0);
    int prev_group = -1;
    for (int li = 0; li < T * BH; ++li) {
      int tile = -1, head = -1;
      fa::grouped_tile_head(li, T, BH, hg, &tile, &head);
      if (tile < 0 || tile >= T || head < 0 || head >= BH) { std::printf("range %d %d %d %d\n", T, BH, hg, li); return 1; }
      if (seen[static_cast<size_t>(tile) * BH + head]++) { std::printf("dup %d %d %d %d\n", T, BH, hg, li); return 1; }
      const int g = head / hg;
      if (g < prev_group) { std::printf("group order %d %d %d\n", T, BH, hg); return 1; }
      prev_group = g;
      // within a group, positions are tile-major: every head of the group gets tile t
      // before any gets tile t + 1
      const int gs = (BH - g * hg) < hg ? (BH - g * hg) : hg;
      const int r = li - g * hg * T;
      if (tile != r / gs) { std::printf("tile order %d %d %d %d\n", T, BH, hg, li); return 1; }
    }
  }
  // head_group: about 32 MiB of Q, K, V, dO per group, within [1, BH]
  struct Case { int BH, Nq, Nk, d, want; };
  const Case cases[] = {{32, 32768, 32768, 128, 1}, {32, 8192, 8192, 128, 4}, {32, 4096, 4096, 128, 8},
                        {32, 1024, 1024, 64, 32}, {3, 100, 100, 32, 3}, {512, 1, 8192, 128, 7}};  // 4 (1 + 8192) 128 bytes a head: 7 fit
  for (const Case& c : cases) {
    const int g = fa::head_group(c.BH, c.Nq, c.Nk, c.d);
    if (g != c.want) { std::printf("head_group %d %d %d %d -> %d\n", c.BH, c.Nq, c.Nk, c.d, g); return 1; }
  }
  std::printf("ok\n");
  return 0;
}
"""


def _cuda_include():
    for cand in ("/usr/local/cuda/include", os.path.join(os.environ.get("CUDA_HOME", ""), "include")):
        if cand and os.path.exists(os.path.join(cand, "cuda_runtime.h")):
            return cand
    return None


def test_launch_order_and_group_size(tmp_path):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "order.cpp"
    src.write_text(CHECKER)
    exe = tmp_path / "order"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", inc, str(src), "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
