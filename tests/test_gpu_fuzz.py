"""Seeded random problems through the CUDA path against the fp64 oracle.

Each case draws a layout (batch, packed varlen, padded varlen with separate
key lengths), a mask kind with a random window, a GQA group, a head-dim pair
the tensor-core kernels take, a 16-bit dtype and a dQ mode, with lengths that
are mostly off the 64/128-row tiles.  Further generators draw the attention
bias shape and dropout probability, fp32 problems for the CUDA-core path
(head dims up to 64, odd d_v), and strided layouts.  The comparison is element
by element and per segment, as in the other parity tests.
"""
import numpy as np
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from tests.test_gpu_extras import run_extras
from tests.test_gpu_parity import B, run_backward_vs_oracle  # noqa: F401  (fixture)
from tests.parity import STRIDED_LAYOUTS, assert_all_ok

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


def _mask(rng, right_max=100, left_max=300):
    mask = int(rng.integers(0, 4))
    left = int(rng.integers(0, left_max)) if mask == 3 else -1
    right = int(rng.choice([-1, 0, int(rng.integers(0, right_max))])) if mask == 3 else -1
    return mask, left, right


def _extras_case(i):
    rng = np.random.default_rng(50000 + i)
    dqk, dv = DIMS[int(rng.integers(0, len(DIMS)))]
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float16
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.choice([1, 2, 4]))
    mask, left, right = _mask(rng)
    wl = W.Workload(f"fuzz_extras{i}", dtype, int(rng.integers(1, 3)), hq, hkv, int(rng.integers(1, 300)),
                    int(rng.integers(1, 300)), dqk, dv, mask, left, right, False, int(rng.integers(0, 2**31 - 1)))
    kind = [None, "11SS", "1HSS", "BHSS", "B1SS"][int(rng.integers(0, 5))]
    p = [0.0, 0.1, 0.25, 0.5][int(rng.integers(0, 4))]
    if kind is None and p == 0.0:
        kind = "BHSS"
    det = int(rng.integers(0, 3))
    return wl, det, kind, p, int(rng.integers(0, 2**40)), int(rng.integers(0, 2**40))


@pytest.mark.parametrize("i", range(60))
def test_random_bias_dropout(B, i):
    wl, det, kind, p, seed, offset = _extras_case(i)
    assert_all_ok(run_extras(B, wl, det, bias_kind=kind, dropout_p=p, seed=seed, offset=offset),
                  f"case {i}: {wl} det={det} bias={kind} p={p}")


def _fp32_case(i):
    rng = np.random.default_rng(70000 + i)
    d, dv = int(rng.choice([4, 8, 16, 32, 64])), int(rng.integers(1, 65))
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.choice([1, 2]))
    mask, left, right = _mask(rng, 50, 100)
    seed = int(rng.integers(0, 2**31 - 1))
    if rng.random() < 0.5:
        wl = W.Workload(f"fuzz_fp32_{i}", torch.float32, int(rng.integers(1, 3)), hq, hkv,
                        int(rng.integers(1, 150)), int(rng.integers(1, 150)), d, dv, mask, left, right, False, seed)
    else:
        nseg = int(rng.integers(1, 4))
        lq = [int(rng.integers(0, 120)) for _ in range(nseg)]
        lq[0] = max(lq[0], 1)
        wl = W.thd(f"fuzz_fp32_{i}", lq, hq=hq, hkv=hkv, d_qk=d, d_v=dv, mask=mask, left=left, right=right,
                   seed=seed, dtype=torch.float32, seqlens_k=[int(rng.integers(0, 120)) for _ in range(nseg)])
    return wl, int(rng.integers(0, 3))


@pytest.mark.parametrize("i", range(40))
def test_random_fp32(B, i):
    wl, det = _fp32_case(i)
    assert_all_ok(run_backward_vs_oracle(B, wl, det), f"case {i}: {wl} det={det}")


@pytest.mark.parametrize("i", range(30))
def test_random_strided_layout(B, i):
    """Batch-mode cases of the first generator in the heads-outer, SBHD and
    packed-QKV layouts (packed only where d_qk == d_v and Sq == Sk)."""
    j = 2000 + i
    wl, det = _case(j)
    while wl.group_mode:
        j += 1000
        wl, det = _case(j)
    layout = STRIDED_LAYOUTS[i % len(STRIDED_LAYOUTS)]
    if layout.__name__ == "layout_packed" and (wl.d_qk != wl.d_v or wl.sq != wl.sk):
        layout = STRIDED_LAYOUTS[0]
    assert_all_ok(run_extras(B, wl, det, layout=layout), f"case {i}: {wl} det={det} layout={layout.__name__}")
