"""The attention cores' launch order (WorkOrder in csrc/attn.cuh) is host logic
shared with the kernels: CTA index -> (batch-head unit, causal-work rank).  Every
CTA index must map to a distinct (unit, rank) pair, so that each block of each
head is computed exactly once, and inside a group the ranks must come heaviest
first.  The header is compiled for the host here (nvcc, no GPU) and the mapping
is checked over many shapes, including a leftover group and a single group."""
import os
import subprocess

import pytest

from tensor_transformer_block_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "tensor_transformer_block_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "attn.cuh"
int main() {
  const int sms_list[3] = {152, 16, 1};
  for (int si = 0; si < 3; ++si)
    for (int units = 1; units <= 70; units += 3)
      for (int blocks = 1; blocks <= 40; blocks += 3) {
        const tpb::WorkOrder o = tpb::make_work_order(units, blocks, sms_list[si]);
        if (o.group < 1 || o.group > units) { printf("bad group %d\n", o.group); return 1; }
        static unsigned char seen[70 * 40];
        for (int i = 0; i < units * blocks; ++i) seen[i] = 0;
        int prev_rank = -1, prev_base = -1;
        for (int idx = 0; idx < o.ctas(); ++idx) {
          int unit, rank;
          o.decode(idx, unit, rank);
          if (unit < 0 || unit >= units || rank < 0 || rank >= blocks) {
            printf("out of range: units %d blocks %d idx %d -> %d %d\n", units, blocks, idx, unit, rank);
            return 1;
          }
          if (seen[unit * blocks + rank]++) { printf("twice: %d %d\n", unit, rank); return 1; }
          // within a group the rank never decreases from one CTA to the next
          const int first = units % o.group;
          const int base = unit < first ? 0 : first + (unit - first) / o.group * o.group;
          if (base == prev_base && rank < prev_rank) { printf("rank order %d %d\n", prev_rank, rank); return 1; }
          prev_base = base;
          prev_rank = rank;
        }
      }
  printf("ok\n");
  return 0;
}
"""


def test_work_order_is_a_heaviest_first_bijection(tmp_path):
    try:
        nvcc = B.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = tmp_path / "work_order.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "work_order"
    r = subprocess.run([nvcc, "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
