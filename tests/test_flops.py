"""The benchmark's mask-adjusted FLOP count against the oracle's own mask
(brute force over the dense visibility matrix), plus the published shapes."""
import pytest

from head_attention_backward_gb300 import flops, workloads
from oracle import attn_ref as R


@pytest.mark.parametrize("lq,lk,m,l,r", [(64, 64, 0, -1, -1), (300, 300, 1, -1, 0), (100, 300, 2, -1, 0),
                                         (300, 100, 2, -1, 0), (500, 500, 3, 100, 0), (90, 120, 3, 30, 20),
                                         (1, 1, 1, -1, 0), (0, 5, 1, -1, 0)])
def test_pairs_match_oracle_mask(lq, lk, m, l, r):
    assert flops.visible_pairs(lq, lk, m, l, r) == R.visible_pairs(lq, lk, m, l, r)


def test_known_workload_flops():
    # causal S=4096: S(S+1)/2 pairs per head; 64 query heads; 2*(3*128+2*128) per pair
    assert flops.bwd_flops(workloads.gqa_causal_det()) == 2 * 32 * 4096 * 4097 / 2 * 2 * 640
    assert abs(flops.bwd_flops(workloads.mha_causal()) - 1.719e11) / 1.719e11 < 1e-3
    w = workloads.window_192()
    pairs = sum(min(i, 1024) + 1 for i in range(8192))
    assert flops.bwd_flops(w) == 16 * pairs * 2 * (3 * 192 + 2 * 128)


def test_thd_segments_fill_exactly():
    segs = workloads.random_segments(16384, 2048, seed=4)
    assert sum(segs) == 16384 and min(segs) >= 1 and max(segs) <= 2048
    assert segs == workloads.random_segments(16384, 2048, seed=4)
