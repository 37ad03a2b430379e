"""The dropout mask code of the kernels (fa_philox.cuh) compiled for the
host, against the float64 oracle's mask (its own Philox4x32-10 and keep
rule): the forward's drop_words (a quad lane's words) and drop_apply (a
quad's words to the 16-bit masks of a row's packed weights), and the
backward's drop_words16 with the row walk (row_key_mask, the dQ pass: 64
keys of a query row) and the column walk (col_query_bits, the dK/dV pass:
64 queries of a key column, as element masks and as the 16-bit pair masks
of the packed P^T), and the one-pass backward's drop_words8 (32 queries of
a key column).

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
#include <cstring>
#include <vector>
#include <cuda_runtime.h>
#include "fa_philox.cuh"
// argv: mode (fwd | row | col) bh seed offset t rows keys; prints the mask,
// one line of 0/1 per row.
int main(int argc, char** argv) {
  const char* mode = argv[1];
  const uint32_t bh = std::strtoul(argv[2], 0, 10);
  const unsigned long long seed = std::strtoull(argv[3], 0, 10);
  const uint32_t off = std::strtoul(argv[4], 0, 10), t = std::strtoul(argv[5], 0, 10);
  const int rows = std::atoi(argv[6]), keys = std::atoi(argv[7]);
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  std::vector<char> m(static_cast<size_t>(rows) * keys, '?');
  auto at = [&](int q, int k) -> char& { return m[static_cast<size_t>(q) * keys + k]; };
  if (!std::strcmp(mode, "fwd")) {
    for (int q = 0; q < rows; ++q)
      for (int key0 = 0; key0 < keys; key0 += 128) {
        uint4 y[4];
        for (uint32_t k = 0; k < 4; ++k)
          y[k] = fa::drop_words(static_cast<uint32_t>(q & ~3), key0, k, bh, off, k0, k1, t);
        uint32_t pk[64];
        for (int i = 0; i < 64; ++i) pk[i] = 0xFFFFFFFFu;
        fa::drop_apply(pk, y, static_cast<uint32_t>(q & 3));
        for (int i = 0; i < 64; ++i) {
          if (pk[i] != 0u && pk[i] != 0xFFFFu && pk[i] != 0xFFFF0000u && pk[i] != 0xFFFFFFFFu) return 2;
          at(q, key0 + 2 * i) = (pk[i] & 0xFFFFu) ? '1' : '0';
          at(q, key0 + 2 * i + 1) = (pk[i] >> 16) ? '1' : '0';
        }
      }
  } else if (!std::strcmp(mode, "row")) {   // dQ pass: query row q, 64 keys from key0
    for (int q = 0; q < rows; ++q)
      for (int key0 = 0; key0 < keys; key0 += 64) {
        uint2 w[4];
        for (uint32_t k = 0; k < 4; ++k)
          w[k] = fa::drop_words16<false>(key0 >> 2, q >> 2, k, bh, off, k0, k1, t);
        for (int b = 0; b < 16; ++b) {
          const uint32_t y = (b >> 3) ? w[b & 3].y : w[b & 3].x;
          for (int c = 0; c < 4; ++c) {
            const uint32_t mk = fa::row_key_mask(y, q & 3, (b >> 2) & 1, c);
            if (mk != 0u && mk != 0xFFFFFFFFu) return 2;
            at(q, key0 + 4 * b + c) = mk ? '1' : '0';
          }
        }
      }
  } else if (!std::strcmp(mode, "col32")) {   // one-pass backward: 32 queries from q0
    for (int key = 0; key < keys; ++key)
      for (int q0 = 0; q0 < rows; q0 += 32) {
        uint32_t w[4];
        for (uint32_t k = 0; k < 4; ++k)
          w[k] = fa::drop_words8(key >> 2, q0 >> 2, k, bh, off, k0, k1, t);
        const uint32_t csel = 0x4440u + (key & 3);
        for (int b = 0; b < 8; ++b) {
          const uint32_t x = fa::col_query_bits(w[b & 3], csel, b >> 2);
          for (int r = 0; r < 4; ++r) {
            const uint32_t mk = fa::prmt(x, 0u, 0x8888u + 0x1111u * r);
            if (mk != 0u && mk != 0xFFFFFFFFu) return 2;
            at(q0 + 4 * b + r, key) = mk ? '1' : '0';
          }
        }
      }
  } else {   // dK/dV pass: key column key, 64 queries from q0
    for (int key = 0; key < keys; ++key)
      for (int q0 = 0; q0 < rows; q0 += 64) {
        uint2 w[4];
        for (uint32_t k = 0; k < 4; ++k)
          w[k] = fa::drop_words16<true>(key >> 2, q0 >> 2, k, bh, off, k0, k1, t);
        const uint32_t csel = 0x4440u + (key & 3);
        for (int b = 0; b < 16; ++b) {
          const uint32_t y = (b >> 3) ? w[b & 3].y : w[b & 3].x;
          const uint32_t x = fa::col_query_bits(y, csel, (b >> 2) & 1);
          for (int r = 0; r < 4; ++r) {
            const uint32_t mk = fa::prmt(x, 0u, 0x8888u + 0x1111u * r);
            if (mk != 0u && mk != 0xFFFFFFFFu) return 2;
            at(q0 + 4 * b + r, key) = mk ? '1' : '0';
          }
          // the pair masks of the packed P^T agree with the element masks
          const uint32_t lo = fa::prmt(x, 0u, 0x9988u), hi = fa::prmt(x, 0u, 0xBBAAu);
          const auto half = [](uint32_t v, int h) { return (v >> (16 * h)) & 0xFFFFu; };
          for (int r = 0; r < 4; ++r) {
            const uint32_t pm = (r < 2) ? half(lo, r) : half(hi, r - 2);
            if ((pm != 0u) != (at(q0 + 4 * b + r, key) == '1') || (pm != 0u && pm != 0xFFFFu)) return 3;
          }
        }
      }
  }
  for (int q = 0; q < rows; ++q) {
    std::fwrite(&m[static_cast<size_t>(q) * keys], 1, keys, stdout);
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
    (0, 0, 0, 0.1, 64, 256),
    (5, 1234, 7, 0.5, 64, 128),
    (77, 2 ** 40 + 3, 2 ** 31 + 5, 0.3, 128, 384),
    (3, 99, 1, 1.0 / 256.0, 64, 128),      # t = 255: the largest threshold
    (1, 5, 0, 0.99, 64, 128),              # t = 3: nearly everything dropped
]


@pytest.mark.parametrize("mode", ["fwd", "row", "col", "col32"])
@pytest.mark.parametrize("bh,seed,off,p,rows,keys", CASES)
def test_packed_mask_matches_oracle(mask_program, mode, bh, seed, off, p, rows, keys):
    t = oracle.dropout_threshold(p)
    out = subprocess.run([mask_program, mode, str(bh), str(seed), str(off), str(t), str(rows),
                          str(keys)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.returncode
    got = np.array([[c == "1" for c in line] for line in out.stdout.split()], dtype=bool)
    want = oracle.dropout_mask(bh, rows, keys, seed, off, p).astype(bool)
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"first mismatches (row, key): {bad[:5].tolist()}"
