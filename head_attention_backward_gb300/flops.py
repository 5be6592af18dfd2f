"""Mask-adjusted FLOP count of the attention backward (measurement only).

Each visible (query, key) pair of each query head costs the five products
S = Q K^T (d_qk), dP = dO V^T (d_v), dV += P^T dO (d_v), dK += dS^T Q (d_qk)
and dQ = dS K (d_qk): 2 * (3 * d_qk + 2 * d_v) FLOPs.  Pairs are counted
exactly from the mask predicate, one query row at a time.
"""
from __future__ import annotations

import numpy as np

MASK_NONE, MASK_CAUSAL_TOP_LEFT, MASK_CAUSAL_BOTTOM_RIGHT, MASK_WINDOW = 0, 1, 2, 3


def visible_pairs(lq: int, lk: int, mask: int, left: int = -1, right: int = -1) -> int:
    if lq <= 0 or lk <= 0:
        return 0
    if mask == MASK_NONE:
        return lq * lk
    if mask == MASK_CAUSAL_TOP_LEFT:
        off, left, right = 0, -1, 0
    elif mask == MASK_CAUSAL_BOTTOM_RIGHT:
        off, left, right = lk - lq, -1, 0
    else:
        off = lk - lq
    i = np.arange(lq, dtype=np.int64)
    lo = np.zeros(lq, dtype=np.int64) if left < 0 else np.maximum(0, i + off - left)
    hi = np.full(lq, lk - 1, dtype=np.int64) if right < 0 else np.minimum(lk - 1, i + off + right)
    return int(np.maximum(0, hi - lo + 1).sum())


def bwd_flops(wl) -> float:
    """FLOPs of one backward pass of a `workloads.Workload`."""
    per_pair = 2.0 * (3 * wl.d_qk + 2 * wl.d_v)
    if wl.group_mode:
        pairs = sum(visible_pairs(nq, nk, wl.mask, wl.left, wl.right)
                    for nq, nk in zip(wl.seqlens, wl.key_lengths))
    else:
        pairs = wl.batch * visible_pairs(wl.sq, wl.sk, wl.mask, wl.left, wl.right)
    return per_pair * pairs * wl.hq
