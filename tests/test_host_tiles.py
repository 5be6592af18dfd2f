"""Host checks of the tile arithmetic the scheduler and the ordered fold rely
on (CPU only).  A small host program built from ``csrc/common.cuh`` checks
``qtile_range`` and ``first_kv_tile`` against brute force over the mask
predicate ``visible``.  It also checks that the KV tiles reaching a query tile
are consecutive: the ordered fold gives the partial of KV tile kt the rank
kt - first_kv_tile and waits for ranks in turn, so a gap would stall it.
Separately, ``visible`` itself is compared with the oracle's mask matrix."""
import os
import shutil
import subprocess

import pytest
import torch

from oracle import attn_ref as R

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "head_attention_backward_gb300", "csrc")

PROG = r"""
#include <cstdio>
#include "common.cuh"
using namespace attn;

// q tiles [lo, hi) holding a query that sees a key of KV tile kt, by brute force
static void brute_range(const MaskArgs& m, int lq, int lk, int kt, int& lo, int& hi) {
  lo = hi = 0;
  bool any = false;
  for (int i = 0; i < lq; ++i)
    for (int j = kt * BN; j < lk && j < (kt + 1) * BN; ++j)
      if (visible(m, i, j)) {
        const int t = i / BM;
        if (!any) { lo = t; any = true; }
        hi = t + 1;
        break;
      }
}

int main() {
  const int lens[] = {0, 1, 63, 64, 65, 128, 129, 257, 300};
  const int wins[] = {-1, 0, 1, 63, 64, 65, 200};
  long cases = 0, bad = 0;
  for (int lq : lens) for (int lk : lens) for (int mask = 0; mask < 4; ++mask)
  for (int l : wins) for (int r : wins) {
    if (mask != 3 && (l != -1 || r != -1)) continue;
    const MaskArgs m = mask_args(mask, l, r, lq, lk);
    const int nkv = (lk + BN - 1) / BN, ntq = (lq + BM - 1) / BM;
    int lo[8], hi[8];
    for (int kt = 0; kt < nkv; ++kt) {
      int a, b;
      qtile_range(m, lq, lk, kt, a, b);
      brute_range(m, lq, lk, kt, lo[kt], hi[kt]);
      const bool same = (a >= b && lo[kt] >= hi[kt]) || (a == lo[kt] && b == hi[kt]);
      ++cases;
      if (!same && bad++ < 10)
        printf("range lq=%d lk=%d mask=%d win=(%d,%d) kt=%d: [%d,%d) vs brute [%d,%d)\n", lq, lk, mask, l, r, kt,
               a, b, lo[kt], hi[kt]);
    }
    for (int qt = 0; qt < ntq; ++qt) {
      int first = -1, last = -1, count = 0;
      for (int kt = 0; kt < nkv; ++kt)
        if (lo[kt] <= qt && qt < hi[kt]) { if (first < 0) first = kt; last = kt; ++count; }
      const int f = first_kv_tile(m, lq, lk, qt);
      ++cases;
      if ((f != first || (count > 0 && count != last - first + 1)) && bad++ < 10)
        printf("first lq=%d lk=%d mask=%d win=(%d,%d) qt=%d: %d vs brute %d (%d tiles in [%d,%d])\n", lq, lk, mask,
               l, r, qt, f, first, count, first, last);
    }
  }
  printf("CHECK %ld %ld\n", cases, bad);
  // visibility matrices of small problems, for the comparison with the oracle
  const int small[] = {1, 3, 7, 12};
  const int swin[] = {-1, 0, 1, 2, 5};
  for (int lq : small) for (int lk : small) for (int mask = 0; mask < 4; ++mask)
  for (int l : swin) for (int r : swin) {
    if (mask != 3 && (l != -1 || r != -1)) continue;
    const MaskArgs m = mask_args(mask, l, r, lq, lk);
    printf("V %d %d %d %d %d ", lq, lk, mask, l, r);
    for (int i = 0; i < lq; ++i)
      for (int j = 0; j < lk; ++j) putchar(visible(m, i, j) ? '1' : '0');
    putchar('\n');
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def host_output():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc unavailable")
    tmp = os.path.join(ROOT, "head_attention_backward_gb300", "_build")
    os.makedirs(tmp, exist_ok=True)
    src = os.path.join(tmp, "host_tiles.cu")
    exe = os.path.join(tmp, "host_tiles")
    open(src, "w").write(PROG)
    r = subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC, "-I",
                        os.path.join(ROOT, "include"), src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return subprocess.run([exe], capture_output=True, text=True, check=True, timeout=120).stdout


def test_tile_ranges_match_brute_force(host_output):
    check = [line for line in host_output.splitlines() if line.startswith("CHECK")]
    assert len(check) == 1, host_output[-2000:]
    _, cases, bad = check[0].split()
    assert int(cases) > 1000
    assert int(bad) == 0, host_output[:2000]


def test_kernel_mask_predicate_equals_oracle(host_output):
    n = 0
    for line in host_output.splitlines():
        if not line.startswith("V "):
            continue
        _, lq, lk, mask, left, right, bits = line.split()
        lq, lk, mask, left, right = map(int, (lq, lk, mask, left, right))
        got = torch.tensor([c == "1" for c in bits], dtype=torch.bool).view(lq, lk)
        want = R.visible(lq, lk, mask, left, right)
        assert torch.equal(got, want), (lq, lk, mask, left, right)
        n += 1
    assert n > 400
