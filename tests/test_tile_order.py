"""The CTA -> (batch-head, tile) order of the kernels (cta_tile in csrc/masks.cuh)
and the host rule that picks its group width (tile_group in csrc/kernels.h),
exercised on the CPU: a small host program compiled with nvcc against the
library's own headers checks that every order is a bijection onto the tiles,
that a group as wide as the tile count is plain head-major order, and that
the width rule gives the groups the kernels are launched with."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_40_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "kernels.h"
#include "masks.cuh"

static int g_sms = 152;
namespace fa {
int sm_count() { return g_sms; }
}

// mode "map": for a grid of shapes, check the order is a bijection and that
// group >= n_tiles reproduces head-major order; print "ok <cases>".
static int check_maps() {
  const int tiles[] = {1, 2, 3, 4, 7, 8, 13, 32, 128, 129};
  const int heads[] = {1, 2, 3, 16, 96, 257};
  const int groups[] = {0, 1, 2, 3, 5, 9, 19, 1000};
  int cases = 0;
  for (int n : tiles)
    for (int BH : heads)
      for (int g0 : groups) {
        const int group = g0 == 1000 ? n : g0;
        std::vector<int> seen(static_cast<size_t>(n) * BH, 0);
        for (int c = 0; c < n * BH; ++c) {
          int bh = -1, rank = -1;
          fa::cta_tile(c, n, BH, group, &bh, &rank);
          if (bh < 0 || bh >= BH || rank < 0 || rank >= n) {
            std::printf("out of range n=%d BH=%d group=%d cta=%d -> %d %d\n", n, BH, group, c,
                        bh, rank);
            return 1;
          }
          if (seen[static_cast<size_t>(bh) * n + rank]++) {
            std::printf("twice n=%d BH=%d group=%d cta=%d\n", n, BH, group, c);
            return 1;
          }
          if (group >= n && (bh != c / n || rank != c % n)) {
            std::printf("not head-major n=%d BH=%d cta=%d\n", n, BH, c);
            return 1;
          }
        }
        ++cases;
      }
  std::printf("ok %d\n", cases);
  return 0;
}

// mode "first": BH heads, n tiles, group w: the largest rank among the first
// w * BH CTAs, and how many heads appear there.
static int first_group(int n, int BH, int w) {
  int max_rank = -1;
  std::vector<int> head(BH, 0);
  for (int c = 0; c < w * BH && c < n * BH; ++c) {
    int bh, rank;
    fa::cta_tile(c, n, BH, w, &bh, &rank);
    if (rank > max_rank) max_rank = rank;
    head[bh] = 1;
  }
  int heads = 0;
  for (int h : head) heads += h;
  std::printf("%d %d\n", max_rank, heads);
  return 0;
}

int main(int argc, char** argv) {
  if (argc >= 2 && std::string(argv[1]) == "map") return check_maps();
  if (argc == 5 && std::string(argv[1]) == "first")
    return first_group(std::atoi(argv[2]), std::atoi(argv[3]), std::atoi(argv[4]));
  if (argc == 8 && std::string(argv[1]) == "group") {
    g_sms = std::atoi(argv[2]);
    std::printf("%d\n", fa::tile_group(std::atoi(argv[3]) != 0, std::atoi(argv[4]),
                                       std::atoi(argv[5]), std::atoi(argv[6]),
                                       std::atoll(argv[7])));
    return 0;
  }
  return 2;
}
"""


@pytest.fixture(scope="module")
def prog(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("tile_order")
    src = d / "tile_order.cu"
    src.write_text(PROGRAM)
    exe = d / "tile_order"
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + os.path.join(ROOT, "include"), "-I" + CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    return str(exe)


def run(prog, *args):
    r = subprocess.run([prog] + [str(a) for a in args], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout.split()


def test_every_order_is_a_bijection_and_full_groups_are_head_major(prog):
    out = run(prog, "map")
    assert out[0] == "ok" and int(out[1]) == 10 * 6 * 8


def test_first_group_holds_the_longest_tiles_of_every_head(prog):
    # 16 heads of 128 query blocks in groups of 19: the first 304 CTAs are
    # ranks 0..18 of all 16 heads.
    assert run(prog, "first", 128, 16, 19) == ["18", "16"]
    # a group as wide as the tile count is head-major: the first 128 x 16
    # CTAs hold every rank
    assert run(prog, "first", 128, 16, 128)[0] == "127"


@pytest.mark.parametrize("args, expected", [
    # (SMs, causal, n_tiles, BH, CTAs per SM, bytes streamed per head)
    ((152, 0, 128, 16, 2, 4 * 16384 * 128), 128),   # not causal: head-major
    ((152, 1, 128, 16, 2, 4 * 16384 * 128), 19),    # 16K forward, two CTAs per SM
    ((152, 1, 128, 16, 1, 4 * 16384 * 128), 9),     # 16K backward, one CTA per SM
    ((152, 1, 8, 96, 2, 4 * 1024 * 64), 3),         # GPT-2-shaped forward
    ((152, 1, 8, 96, 1, 4 * 1024 * 64), 1),         # GPT-2-shaped backward: 25 MB fits
    ((152, 1, 16, 128, 1, 4 * 2048 * 128), 16),     # 2K, 128 heads, d = 128: 128 MB, head-major
    ((152, 1, 4, 16, 2, 4 * 512 * 64), 4),          # width capped at the tile count
    ((0, 1, 4, 16, 2, 4 * 512 * 64), 1),            # SM count unknown: still a valid order
])
def test_group_width_rule(prog, args, expected):
    assert int(run(prog, "group", *args)[0]) == expected
