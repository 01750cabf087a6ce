"""CPU checks of the logic the kernels and the host share (csrc/fa_params.h,
compiled with the host compiler into small programs; no GPU):

`wave_order`, for every unit count up to 700 and every grid up to 160:
* slot -> unit is a bijection of [0, num_units) (no unit skipped or run
  twice, whatever the partial last wave);
* even waves keep their order and full odd waves are reversed (CTA 0 takes
  the last unit of an odd wave);
* on a heaviest-first list of causal unit costs (pair p of a head costs
  2p + 2.5 key steps, 32 heads), the busiest CTA's total is within 3 % of
  the mean, where taking the slots in order leaves it 10 % above.

`key_tile_range` (the block skipping of every kernel), against brute force
over small problems: the key tiles [n0, n1) it returns for a block of rows
are exactly the tiles holding a key that some row of the block may see
(row i sees keys i - win_left .. i + win_right below N).

`clip_to_split`: the split's tile range is the intersection of the tiles
with the split's own, empty when they do not meet.

`packed_rows` (offsets and used lengths of packed batches), on random and
malformed offsets: the rows it returns always lie inside [0, total), the
length never exceeds the cap, the used length or the offsets' difference,
and well-formed offsets come back unchanged.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_forward_10_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include "fa_params.h"
#include <algorithm>
#include <cstdio>
#include <vector>

static double busiest_over_mean(const std::vector<double>& cost, int grid, bool alternate) {
  const int n = static_cast<int>(cost.size());
  std::vector<double> cta(grid, 0.0);
  double total = 0.0;
  for (int s = 0; s < n; ++s) {
    const int u = alternate ? fa::wave_order(s, n, grid) : s;
    cta[s % grid] += cost[u];
    total += cost[u];
  }
  return *std::max_element(cta.begin(), cta.end()) / (total / grid);
}

int main() {
  long bad_bijection = 0, bad_order = 0;
  for (int n = 1; n <= 700; ++n)
    for (int g = 1; g <= 160; ++g) {
      std::vector<int> seen(n, 0);
      for (int s = 0; s < n; ++s) {
        const int u = fa::wave_order(s, n, g);
        if (u < 0 || u >= n || seen[u]++) ++bad_bijection;
        const int k = s / g, c = s % g;
        const bool full = (k + 1) * g <= n;
        if (k % 2 == 0 && u != s) ++bad_order;
        if (k % 2 == 1 && full && u != k * g + (g - 1 - c)) ++bad_order;
      }
    }
  // causal pair units of 32 heads, 32 pairs per head, heaviest first
  std::vector<double> cost;
  for (int pe = 0; pe < 32; ++pe)
    for (int h = 0; h < 32; ++h) cost.push_back(2.0 * (31 - pe) + 2.5);
  // key_tile_range against brute force
  long bad_range = 0;
  for (int N = 1; N <= 70; N += 3)
    for (int tile : {8, 16})
      for (int wl : {0, 1, 5, 17, 200})
        for (int wr : {0, 3, 9, 200})
          for (int r0 = 0; r0 < N; r0 += 2)
            for (int r_end = r0 + 1; r_end <= std::min(N + 9, r0 + 20); r_end += 3) {
              int n0, n1;
              fa::key_tile_range(r0, r_end, N, wl, wr, tile, &n0, &n1);
              const int tiles = (N + tile - 1) / tile;
              for (int t = 0; t < tiles + 1; ++t) {
                bool any = false;
                for (int j = t * tile; j < std::min(N, (t + 1) * tile); ++j)
                  for (int i = r0; i < r_end && !any; ++i)
                    if (j >= i - wl && j <= i + wr) any = true;
                const bool in = t >= n0 && t < n1;
                if (any != in) ++bad_range;
              }
            }
  // clip_to_split
  long bad_clip = 0;
  for (int a = 0; a < 12; ++a)
    for (int b = a; b < 12; ++b)
      for (int st = 1; st < 6; ++st)
        for (int s = 0; s < 6; ++s) {
          int n0 = a, n1 = b;
          fa::clip_to_split(s, st, &n0, &n1);
          const int lo = std::max(a, s * st), hi = std::min(b, (s + 1) * st);
          if (hi > lo ? (n0 != lo || n1 != hi) : (n1 != n0)) ++bad_clip;
        }
  // packed_rows on random (often malformed) offsets
  long bad_rows = 0;
  unsigned seed = 12345u;
  auto rnd = [&](int m) { seed = seed * 1103515245u + 12345u; return static_cast<int>((seed >> 8) % m); };
  for (int trial = 0; trial < 20000; ++trial) {
    const int batch = 1 + rnd(6), total = rnd(300), cap = 1 + rnd(200);
    const bool malformed = rnd(2) == 0;
    std::vector<int> cu(batch + 1), used(batch);
    cu[0] = malformed ? rnd(400) - 50 : 0;
    for (int b = 0; b < batch; ++b)
      cu[b + 1] = malformed ? rnd(400) - 50 : std::min(total, cu[b] + rnd(120));
    for (int b = 0; b < batch; ++b) used[b] = rnd(3) == 0 ? rnd(150) - 10 : 1 << 30;
    const bool with_used = rnd(2) == 0;
    for (int b = 0; b < batch; ++b) {
      int first, len;
      fa::packed_rows(cu.data(), with_used ? used.data() : nullptr, b, total, cap, &first, &len);
      if (first < 0 || first > total || len < 0 || first + len > total || len > cap) ++bad_rows;
      if (with_used && len > std::max(0, used[b])) ++bad_rows;
      if (!malformed && !with_used &&
          (first != cu[b] || len != std::min(cap, cu[b + 1] - cu[b]))) ++bad_rows;
    }
  }
  std::printf("%ld %ld %.4f %.4f %ld %ld %ld\n", bad_bijection, bad_order,
              busiest_over_mean(cost, 152, false), busiest_over_mean(cost, 152, true),
              bad_range, bad_clip, bad_rows);
  return 0;
}
"""


def _run_program(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "wave_order.cc"
    exe = tmp_path / "wave_order"
    src.write_text(PROGRAM)
    subprocess.run([gxx, "-std=c++17", "-O2", "-D__host__=", "-D__device__=",
                    "-D__forceinline__=inline", f"-I{CSRC}", f"-I{CUDA_INC}", str(src), "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    return subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    return _run_program(tmp_path_factory.mktemp("host_logic"))


def test_wave_order(results):
    bad_bijection, bad_order = int(results[0]), int(results[1])
    in_order, alternating = float(results[2]), float(results[3])
    assert bad_bijection == 0 and bad_order == 0
    assert in_order > 1.10, in_order
    assert alternating < 1.03, alternating


def test_key_tile_range_matches_brute_force(results):
    assert int(results[4]) == 0


def test_clip_to_split(results):
    assert int(results[5]) == 0


def test_packed_rows_stay_in_bounds(results):
    assert int(results[6]) == 0
