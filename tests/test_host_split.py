"""Host logic of the forward's work split, compiled from the shared header
(no GPU): the unit order `ra::unit_coords` visits every (query-tile pair,
batch, query head) exactly once for any block size, reduces to pair-major
order with heads innermost for blocks of one pair, and with blocks of
G / (Hq / Hkv) pairs puts a single key/value stream into each round of G
units."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "blockwise_attention_online_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <cuda_runtime.h>
#include <cstdio>
#include <set>
#include <tuple>
#include "ra_plan.h"

static int check(int npairs, int B, int Hq, int Hkv, int P) {
  std::set<std::tuple<int, int, int>> seen;
  const int units = npairs * B * Hq;
  for (int u = 0; u < units; ++u) {
    int rank, b, hq;
    ra::unit_coords(u, npairs, B, Hq, Hkv, P, rank, b, hq);
    if (rank < 0 || rank >= npairs || b < 0 || b >= B || hq < 0 || hq >= Hq) return 1;
    if (!seen.insert(std::make_tuple(rank, b, hq)).second) return 2;
    if (P == 1) {
      const int BH = B * Hq;
      if (rank != u / BH || b * Hq + hq != u % BH) return 3;
    }
  }
  return int(seen.size()) == units ? 0 : 4;
}

int main() {
  const int shapes[][5] = {{512, 1, 32, 8, 38}, {512, 2, 32, 8, 38}, {7, 3, 6, 2, 3},
                           {100, 1, 16, 1, 9},  {5, 1, 8, 8, 1},    {13, 2, 4, 2, 13},
                           {9, 2, 8, 2, 1},     {128, 1, 32, 32, 1}, {33, 1, 12, 3, 50}};
  for (const auto& s : shapes) {
    const int P = s[4] < s[0] ? s[4] : s[0];
    const int r = check(s[0], s[1], s[2], s[3], P);
    if (r) { std::printf("fail %d %d %d %d %d: %d\n", s[0], s[1], s[2], s[3], P, r); return 1; }
  }
  // 131072 rows (512 pairs), 32 query heads on 8 key/value heads, 152 CTAs:
  // blocks of 152 / 4 = 38 pair ranks make every round one key/value stream
  for (int round = 0; round < 512 * 32 / 152; ++round) {
    std::set<int> streams;
    for (int c = 0; c < 152; ++c) {
      int rank, b, hq;
      ra::unit_coords(round * 152 + c, 512, 1, 32, 8, 38, rank, b, hq);
      streams.insert(b * 8 + hq / 4);
    }
    if (round < 13 * 8 && streams.size() != 1) { std::printf("round %d: %zu streams\n", round, streams.size()); return 1; }
  }
  std::printf("ok\n");
  return 0;
}
"""


def test_unit_order_visits_every_unit_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.isdir(CUDA_INC):
        pytest.skip("needs a C++ compiler and the CUDA headers")
    src = tmp_path / "unit_order.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "unit_order"
    subprocess.check_call([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                           "-I", CUDA_INC, str(src), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
