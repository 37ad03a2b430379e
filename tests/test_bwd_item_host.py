"""The backward kernels' deal of work items (bwd_item in fa_bwd_kernel.cuh),
compiled for the host: items come in groups of item_group heads, tile by
tile within a group, the last group possibly smaller.  For every shape
below, the items 0 .. BH * n - 1 must map one to one onto the (tile, head)
pairs, each group must hold its own heads, and inside a group the tile
index must never decrease (the heaviest tiles of causal calls first)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_14_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r'''
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "fa_bwd_kernel.cuh"
// argv: BH n group; prints "ok" or the first violation.
int main(int argc, char** argv) {
  const int BH = std::atoi(argv[1]), n = std::atoi(argv[2]), G = std::atoi(argv[3]);
  fa::BwdParams p{};
  p.BH = BH;
  p.item_group = G;
  std::vector<int> seen(static_cast<size_t>(BH) * n, 0);
  int prev_tile = -1, prev_group = -1;
  for (int item = 0; item < BH * n; ++item) {
    int tile = -1, bh = -1;
    fa::bwd_item(p, item, n, tile, bh);
    if (tile < 0 || tile >= n || bh < 0 || bh >= BH) { std::printf("range %d\n", item); return 1; }
    if (seen[static_cast<size_t>(bh) * n + tile]++) { std::printf("twice %d\n", item); return 1; }
    const int group = bh / G;
    if (group != item / (G * n)) { std::printf("group %d\n", item); return 1; }
    if (group == prev_group && tile < prev_tile) { std::printf("order %d\n", item); return 1; }
    prev_tile = tile;
    prev_group = group;
  }
  std::printf("ok\n");
  return 0;
}
'''


@pytest.fixture(scope="module")
def item_program(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc) and not shutil.which("nvcc"):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("item")
    src, exe = d / "item.cu", d / "item"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", CSRC, "-I", INCLUDE, str(src), "-o", str(exe)], check=True,
                   capture_output=True, timeout=600)
    return str(exe)


@pytest.mark.parametrize("BH,n,G", [(1, 1, 1), (16, 32, 1), (12, 5, 8), (10, 16, 8), (8, 256, 8),
                                    (128, 64, 8), (3, 7, 3), (256, 8, 1), (13, 3, 4)])
def test_items_cover_every_pair_once(item_program, BH, n, G):
    out = subprocess.run([item_program, str(BH), str(n), str(G)], capture_output=True, text=True,
                         timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
