"""Seeded synthetic inputs for the FMHA backward workloads.

This module holds no attention arithmetic: only shapes, seeds and random
draws, so that the CUDA path and the fp64 oracle can be fed identical bits.
Tensors are drawn on the CPU from ``torch.Generator`` in fp32 ~ N(0, 1) and
cast to the workload dtype there; callers copy them to the device.

The workloads stand in for the packed-document Llama-3-8B-shaped traffic of
the TransformerEngine THD fix (PR #671, Verification): GQA with 32 query and
8 kv heads, head dim 128, causal masks within each packed segment.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

MASK_NONE, MASK_CAUSAL_TOP_LEFT, MASK_CAUSAL_BOTTOM_RIGHT, MASK_WINDOW = 0, 1, 2, 3


@dataclasses.dataclass
class Workload:
    name: str
    dtype: torch.dtype
    batch: int            # B in batch mode; number of segments in group mode
    hq: int
    hkv: int
    sq: int               # batch: sequence length; group: max segment length
    sk: int
    d_qk: int
    d_v: int
    mask: int
    left: int = -1
    right: int = -1
    deterministic: bool = False
    seed: int = 0
    seqlens: Optional[List[int]] = None   # group (THD) mode when set

    @property
    def group_mode(self) -> bool:
        return self.seqlens is not None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_qk)

    @property
    def total(self) -> int:
        return sum(self.seqlens) if self.group_mode else self.batch * self.sq

    def cu_seqlens(self) -> Optional[torch.Tensor]:
        if not self.group_mode:
            return None
        cu = [0]
        for n in self.seqlens:
            cu.append(cu[-1] + n)
        return torch.tensor(cu, dtype=torch.int32)

    def shapes(self):
        if self.group_mode:
            t = self.total
            return dict(q=(t, self.hq, self.d_qk), k=(t, self.hkv, self.d_qk),
                        v=(t, self.hkv, self.d_v), o=(t, self.hq, self.d_v),
                        lse=(self.hq, t))
        b = self.batch
        return dict(q=(b, self.sq, self.hq, self.d_qk), k=(b, self.sk, self.hkv, self.d_qk),
                    v=(b, self.sk, self.hkv, self.d_v), o=(b, self.sq, self.hq, self.d_v),
                    lse=(b, self.hq, self.sq))

    def inputs(self):
        """Q, K, V, dO ~ N(0, 1) in the workload dtype (CPU tensors)."""
        g = torch.Generator().manual_seed(self.seed)
        sh = self.shapes()
        out = {}
        for name in ("q", "k", "v", "do"):
            shape = sh["o"] if name == "do" else sh[name]
            out[name] = torch.randn(shape, generator=g, dtype=torch.float32).to(self.dtype)
        return out


def random_segments(total: int, max_len: int, seed: int) -> List[int]:
    """Segment lengths drawn uniformly from [1, max_len] until `total` is reached;
    the last segment is trimmed so the lengths sum to exactly `total`."""
    rng = np.random.default_rng(seed)
    out: List[int] = []
    acc = 0
    while acc < total:
        n = int(rng.integers(1, max_len + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def thd(name: str, seqlens: List[int], hq=32, hkv=8, d_qk=128, d_v=128,
        mask=MASK_CAUSAL_TOP_LEFT, left=-1, right=-1, deterministic=False, seed=3,
        dtype=torch.bfloat16) -> Workload:
    mx = max(seqlens) if seqlens else 0
    return Workload(name, dtype, len(seqlens), hq, hkv, mx, mx, d_qk, d_v, mask, left, right,
                    deterministic, seed, list(seqlens))


# The five workloads of the benchmark specification.
def tiny_fp32() -> Workload:
    return Workload("tiny_fp32_B1_H2_S64_d32", torch.float32, 1, 2, 2, 64, 64, 32, 32,
                    MASK_NONE, seed=0)


def mha_causal() -> Workload:
    return Workload("mha_B4_H16_S2048_d128_causal", torch.bfloat16, 4, 16, 16, 2048, 2048,
                    128, 128, MASK_CAUSAL_TOP_LEFT, seed=1)


def gqa_causal_det() -> Workload:
    return Workload("gqa_B2_Hq32_Hkv8_S4096_d128_causal_det", torch.bfloat16, 2, 32, 8,
                    4096, 4096, 128, 128, MASK_CAUSAL_TOP_LEFT, deterministic=True, seed=2)


def thd_packed(deterministic=False) -> Workload:
    segs = random_segments(16384, 2048, seed=4)
    return thd("thd_T16384_Hq32_Hkv8_d128_causal", segs, deterministic=deterministic, seed=3)


def window_192(deterministic=True) -> Workload:
    return Workload("win_B1_H16_S8192_dqk192_dv128_left1024", torch.bfloat16, 1, 16, 16,
                    8192, 8192, 192, 128, MASK_WINDOW, left=1024, right=0,
                    deterministic=deterministic, seed=5)


# Fixed splits the THD fix was verified on (PR #671, Verification and the
# review reply on non-16-multiple lengths).
PAGE_SPLITS = [[256], [100, 80, 76], [128, 128], [64, 64, 64, 64], [200, 56], [103, 77, 61]]
