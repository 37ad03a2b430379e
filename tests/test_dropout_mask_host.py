"""The forward pass's dropout mask code (fa_philox.cuh: drop_words, which
draws a quad lane's words, and drop_apply, which turns a quad's words into
the 16-bit masks of a row's packed weights) compiled for the host, against
the float64 oracle's mask (its own Philox4x32-10 and keep rule).

The mask is what "Why FlashAttention Can Avoid a Square Attention Array
Without Making Attention Linear", section "Backward can recreate tiles
instead of retaining the square", has the backward pass regenerate from
the kept generator state; a wrong row shift, block order or byte test in
the packed layout shows here as a mismatched key, on the CPU.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_14_gb300", "csrc")

PROGRAM = r'''
#include <cstdio>
#include <cstdlib>
#include <cuda_runtime.h>
#include "fa_philox.cuh"
// argv: bh seed offset t rows keys; prints one line of 0/1 per row.
int main(int argc, char** argv) {
  const uint32_t bh = std::strtoul(argv[1], 0, 10);
  const unsigned long long seed = std::strtoull(argv[2], 0, 10);
  const uint32_t off = std::strtoul(argv[3], 0, 10), t = std::strtoul(argv[4], 0, 10);
  const int rows = std::atoi(argv[5]), keys = std::atoi(argv[6]);
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int q = 0; q < rows; ++q) {
    for (int key0 = 0; key0 < keys; key0 += 128) {
      uint4 y[4];
      for (uint32_t k = 0; k < 4; ++k)
        y[k] = fa::drop_words(static_cast<uint32_t>(q & ~3), key0, k, bh, off, k0, k1, t);
      uint32_t pk[64];
      for (int i = 0; i < 64; ++i) pk[i] = 0xFFFFFFFFu;
      fa::drop_apply(pk, y, static_cast<uint32_t>(q & 3));
      for (int i = 0; i < 64; ++i) {
        if (pk[i] != 0u && pk[i] != 0xFFFFu && pk[i] != 0xFFFF0000u && pk[i] != 0xFFFFFFFFu) return 2;
        std::putchar((pk[i] & 0xFFFFu) ? '1' : '0');
        std::putchar((pk[i] >> 16) ? '1' : '0');
      }
    }
    std::putchar('\n');
  }
  return 0;
}
'''


@pytest.fixture(scope="module")
def mask_program(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc) and not shutil.which("nvcc"):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("mask")
    src, exe = d / "mask.cu", d / "mask"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True, timeout=300)
    return str(exe)


CASES = [
    # bh, seed, offset, p, rows, keys
    (0, 0, 0, 0.1, 8, 256),
    (5, 1234, 7, 0.5, 12, 128),
    (77, 2 ** 40 + 3, 2 ** 31 + 5, 0.3, 4, 384),
    (3, 99, 1, 1.0 / 256.0, 8, 128),       # t = 255: the largest threshold
    (1, 5, 0, 0.99, 8, 128),               # t = 3: nearly everything dropped
]


@pytest.mark.parametrize("bh,seed,off,p,rows,keys", CASES)
def test_packed_mask_matches_oracle(mask_program, bh, seed, off, p, rows, keys):
    t = oracle.dropout_threshold(p)
    out = subprocess.run([mask_program, str(bh), str(seed), str(off), str(t), str(rows), str(keys)],
                         capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.returncode
    got = np.array([[c == "1" for c in line] for line in out.stdout.split()], dtype=bool)
    want = oracle.dropout_mask(bh, rows, keys, seed, off, p).astype(bool)
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"first mismatches (row, key): {bad[:5].tolist()}"
