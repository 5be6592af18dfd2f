"""Seeded random problems through the CUDA path against the fp64 oracle.

Each case draws a layout (batch, packed varlen, padded varlen with separate
key lengths), a mask kind with a random window, a GQA group, a head-dim pair
the tensor-core kernels take, a 16-bit dtype and a dQ mode, with lengths that
are mostly off the 64/128-row tiles.  The comparison is element by element
and per segment, as in the other parity tests.
"""
import numpy as np
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from tests.test_gpu_parity import B, run_backward_vs_oracle  # noqa: F401  (fixture)
from tests.parity import assert_all_ok

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (128, 128), (192, 128), (256, 256)]


def _case(i):
    rng = np.random.default_rng(1000 + i)
    dqk, dv = DIMS[int(rng.integers(0, len(DIMS)))]
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float16
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.choice([1, 2, 4]))
    mask = int(rng.integers(0, 4))
    left = int(rng.integers(0, 300)) if mask == 3 else -1
    right = int(rng.choice([-1, 0, int(rng.integers(0, 100))])) if mask == 3 else -1
    det = int(rng.integers(0, 3))
    layout = int(rng.integers(0, 3))
    seed = int(rng.integers(0, 2**31 - 1))
    if layout == 0:   # batch mode
        sq, sk = int(rng.integers(1, 400)), int(rng.integers(1, 400))
        wl = W.Workload(f"fuzz{i}", dtype, int(rng.integers(1, 3)), hq, hkv, sq, sk, dqk, dv, mask, left, right,
                        False, seed)
    else:             # packed or padded varlen, own key lengths
        nseg = int(rng.integers(1, 5))
        lq = [int(rng.integers(0, 300)) for _ in range(nseg)]
        lk = [int(rng.integers(0, 300)) for _ in range(nseg)]
        if sum(lq) == 0:
            lq[0] = 1
        gq = [int(rng.integers(0, 40)) for _ in range(nseg + 1)] if layout == 2 else None
        gk = [int(rng.integers(0, 40)) for _ in range(nseg + 1)] if layout == 2 else None
        wl = W.thd(f"fuzz{i}", lq, hq=hq, hkv=hkv, d_qk=dqk, d_v=dv, mask=mask, left=left, right=right,
                   seed=seed, dtype=dtype, seqlens_k=lk, gaps_q=gq, gaps_k=gk)
    return wl, det


@pytest.mark.parametrize("i", range(32))
def test_random_problem(B, i):
    wl, det = _case(i)
    assert_all_ok(run_backward_vs_oracle(B, wl, det), f"case {i}: {wl} det={det}")
