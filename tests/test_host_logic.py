"""CPU checks of the scheduling logic the kernels and the host share
(`wave_order` in csrc/fa_params.h): the header is compiled with the host
compiler (no GPU) into a small program that checks, for every unit count up
to 700 and every grid up to 160:

* slot -> unit is a bijection of [0, num_units) (no unit skipped or run
  twice, whatever the partial last wave);
* even waves keep their order and full odd waves are reversed (CTA 0 takes
  the last unit of an odd wave);
* on a heaviest-first list of causal unit costs (pair p of a head costs
  2p + 2.5 key steps, 32 heads), the busiest CTA's total is within 3 % of
  the mean, where taking the slots in order leaves it 10 % above.
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
  std::printf("%ld %ld %.4f %.4f\n", bad_bijection, bad_order,
              busiest_over_mean(cost, 152, false), busiest_over_mean(cost, 152, true));
  return 0;
}
"""


def test_wave_order(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda.h")):
        pytest.skip("needs g++ and the CUDA headers")
    src = tmp_path / "wave_order.cc"
    exe = tmp_path / "wave_order"
    src.write_text(PROGRAM)
    subprocess.run([gxx, "-std=c++17", "-O2", "-D__host__=", "-D__device__=",
                    "-D__forceinline__=inline", f"-I{CSRC}", f"-I{CUDA_INC}", str(src), "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    bad_bijection, bad_order = int(out[0]), int(out[1])
    in_order, alternating = float(out[2]), float(out[3])
    assert bad_bijection == 0 and bad_order == 0
    assert in_order > 1.10, in_order
    assert alternating < 1.03, alternating
