"""Host constants of the forward's division-free unit decoding.

The forward kernel decodes each work unit with divisions by values fixed at
launch (B*H and H) done as a multiply-high and a shift, with constants from
`make_fast_div` in csrc/common.cuh (Granlund and Montgomery, "Division by
Invariant Integers using Multiplication").  This compiles a small host
program against that header and compares the multiply-shift quotient with
the exact integer quotient n / d for every divisor up to 4096, powers of two
and their neighbours and random large divisors, each over edge and random
dividends below 2^31 (the kernels' unit numbers stay below 2^31).  It also
checks that `make_unit_order` splits a launch into whole groups and a last
group that add up to the heads."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_exact_attention_flash_gb300", "csrc")

PROGRAM = r"""
#include "common.cuh"
#include <cstdio>
#include <cstdint>
#include <vector>

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32() {  // xorshift64*, a fixed seed
  state ^= state >> 12;
  state ^= state << 25;
  state ^= state >> 27;
  return uint32_t((state * 0x2545F4914F6CDD1Dull) >> 32);
}

int main() {
  std::vector<uint32_t> ds;
  for (uint32_t d = 1; d <= 4096; ++d) ds.push_back(d);
  for (int k = 1; k < 31; ++k) {
    ds.push_back(1u << k);
    ds.push_back((1u << k) - 1);
    ds.push_back((1u << k) + 1);
  }
  for (int i = 0; i < 2000; ++i) ds.push_back(1 + next_u32() % 0x7FFFFFFFu);
  long checked = 0;
  for (uint32_t d : ds) {
    const fmsa::FastDiv f = fmsa::make_fast_div(d);
    std::vector<uint32_t> ns = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d, 0x7FFFFFFEu, 0x7FFFFFFFu};
    for (int i = 0; i < 200; ++i) ns.push_back(next_u32() & 0x7FFFFFFFu);
    for (int i = 0; i < 50; ++i) {  // either side of a multiple of d
      const uint32_t m = (next_u32() & 0x7FFFFFFFu) / d * d;
      ns.push_back(m);
      if (m > 0) ns.push_back(m - 1);
    }
    for (uint32_t n : ns) {
      if (n > 0x7FFFFFFFu) continue;
      const uint32_t t = uint32_t((uint64_t(n) * f.mul) >> 32);
      const uint64_t sum = uint64_t(t) + n;
      if (sum >> 32) {
        std::printf("overflow d=%u n=%u\n", d, n);
        return 1;
      }
      const uint32_t q = uint32_t(sum) >> f.shift;
      if (q != n / d) {
        std::printf("mismatch d=%u n=%u got %u want %u\n", d, n, q, n / d);
        return 1;
      }
      ++checked;
    }
  }
  const int cases[][4] = {{1, 32, 64, 32}, {4, 16, 32, 64}, {1, 6, 256, 4}, {2, 3, 5, 4}, {1, 1, 2, 1}};
  for (const auto& c : cases) {
    const fmsa::UnitOrder o = fmsa::make_unit_order(c[0], c[1], c[2], c[3]);
    if (o.n_full * o.group + o.last != c[0] * c[1] || o.last < 0 || o.last >= o.group) {
      std::printf("unit order B=%d H=%d group=%d: %d x %d + %d\n", c[0], c[1], c[3], o.n_full,
                  o.group, o.last);
      return 1;
    }
  }
  std::printf("ok %ld\n", checked);
  return 0;
}
"""


def _nvcc():
    found = shutil.which("nvcc")
    if found:
        return found
    default = "/usr/local/cuda/bin/nvcc"
    return default if os.path.exists(default) else None


def test_fast_div_constants_give_exact_quotients(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    src = tmp_path / "fast_div_check.cu"
    exe = tmp_path / "fast_div_check"
    src.write_text(PROGRAM)
    build = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                            str(src), "-o", str(exe)], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr[-2000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.startswith("ok ")
    assert int(run.stdout.split()[1]) > 1_000_000
