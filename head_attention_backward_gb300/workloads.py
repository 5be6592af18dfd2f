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
    seqlens_k: Optional[List[int]] = None # key lengths per segment when they differ from seqlens
    # padded group layout: gaps[g] = padding rows in front of segment g, the
    # last entry after the last segment (nseg + 1 entries); None = packed
    gaps_q: Optional[List[int]] = None
    gaps_k: Optional[List[int]] = None

    @property
    def group_mode(self) -> bool:
        return self.seqlens is not None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_qk)

    @property
    def key_lengths(self) -> Optional[List[int]]:
        if not self.group_mode:
            return None
        return self.seqlens if self.seqlens_k is None else self.seqlens_k

    @property
    def total(self) -> int:
        """Query rows of the tensors (padding rows included)."""
        if not self.group_mode:
            return self.batch * self.sq
        return sum(self.seqlens) + (sum(self.gaps_q) if self.gaps_q else 0)

    @property
    def total_k(self) -> int:
        if not self.group_mode:
            return self.batch * self.sk
        return sum(self.key_lengths) + (sum(self.gaps_k) if self.gaps_k else 0)

    @staticmethod
    def _starts(lengths, gaps) -> torch.Tensor:
        """Physical start row of every segment, then the row total."""
        st, r = [], 0
        for b, n in enumerate(lengths):
            r += gaps[b]
            st.append(r)
            r += n
        st.append(r + gaps[len(lengths)])
        return torch.tensor(st, dtype=torch.int32)

    def cu_seqlens_q_padded(self) -> Optional[torch.Tensor]:
        return self._starts(self.seqlens, self.gaps_q) if self.group_mode and self.gaps_q else None

    def cu_seqlens_k_padded(self) -> Optional[torch.Tensor]:
        return self._starts(self.key_lengths, self.gaps_k) if self.group_mode and self.gaps_k else None

    def padding_rows(self, side: str) -> List[int]:
        """Rows of the q ("q") or k ("k") tensors that belong to no segment."""
        st = self.cu_seqlens_q_padded() if side == "q" else self.cu_seqlens_k_padded()
        if st is None:
            return []
        lens = self.seqlens if side == "q" else self.key_lengths
        inside = set()
        for b, n in enumerate(lens):
            inside.update(range(int(st[b]), int(st[b]) + n))
        total = self.total if side == "q" else self.total_k
        return [r for r in range(total) if r not in inside]

    @staticmethod
    def _offsets(lengths) -> torch.Tensor:
        cu = [0]
        for n in lengths:
            cu.append(cu[-1] + n)
        return torch.tensor(cu, dtype=torch.int32)

    def cu_seqlens(self) -> Optional[torch.Tensor]:
        """Query segment offsets (group mode), else None."""
        return self._offsets(self.seqlens) if self.group_mode else None

    def cu_seqlens_k(self) -> Optional[torch.Tensor]:
        """Key segment offsets (group mode), else None."""
        return self._offsets(self.key_lengths) if self.group_mode else None

    def shapes(self):
        if self.group_mode:
            t, tk = self.total, self.total_k
            return dict(q=(t, self.hq, self.d_qk), k=(tk, self.hkv, self.d_qk),
                        v=(tk, self.hkv, self.d_v), o=(t, self.hq, self.d_v),
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
        dtype=torch.bfloat16, seqlens_k=None, gaps_q=None, gaps_k=None) -> Workload:
    """THD workload; `seqlens_k` gives per-segment key lengths when they differ
    from the query lengths (cross attention); `gaps_q` / `gaps_k` (one entry
    per segment plus one) place padding rows around the segments."""
    if seqlens_k is not None and len(seqlens_k) != len(seqlens):
        raise ValueError("seqlens and seqlens_k need one entry per segment")
    for gaps in (gaps_q, gaps_k):
        if gaps is not None and len(gaps) != len(seqlens) + 1:
            raise ValueError("gaps need one entry per segment plus one")
    mx = max(seqlens) if seqlens else 0
    mk = max(seqlens_k) if seqlens_k else mx
    return Workload(name, dtype, len(seqlens), hq, hkv, mx, mk, d_qk, d_v, mask, left, right,
                    deterministic, seed, list(seqlens),
                    None if seqlens_k is None else list(seqlens_k),
                    None if gaps_q is None else list(gaps_q),
                    None if gaps_k is None else list(gaps_k))


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


def gqa_d256(deterministic=True) -> Workload:
    """Head dim 256 (the widest pair the library takes): GQA, causal."""
    return Workload("gqa_B1_Hq16_Hkv4_S4096_d256_causal", torch.bfloat16, 1, 16, 4, 4096, 4096, 256, 256,
                    MASK_CAUSAL_TOP_LEFT, deterministic=deterministic, seed=6)


# Fixed splits the THD fix was verified on (PR #671, Verification and the
# review reply on non-16-multiple lengths).
PAGE_SPLITS = [[256], [100, 80, 76], [128, 128], [64, 64, 64, 64], [200, 56], [103, 77, 61]]
