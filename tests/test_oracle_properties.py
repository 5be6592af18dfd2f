"""Property-based pins of the oracle (CPU only).

For random small problems -- 1 to 3 packed segments with their own query and
key lengths (zero included), every mask kind with random windows, GQA groups,
head dims and scales -- the oracle's forward and backward equal torch's
scaled_dot_product_attention and its autograd backward, segment by segment.
SDPA shares no code with the oracle.  The mask is written out here from the
predicate the mask enum stands for (key j visible to query i, with
off = Lk - Lq for the bottom-right kinds), not taken from the oracle.  Rows
that see no key are checked against the oracle's reading instead (LSE = -inf,
O = 0, zero gradient), since SDPA returns NaN for them.
"""
import math

import pytest
import torch

pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import attn_ref as R  # noqa: E402

F64 = torch.float64


def mask_matrix(lq, lk, mask, left, right):
    off = 0 if mask in (0, 1) else lk - lq
    if mask in (1, 2):
        left, right = -1, 0
    elif mask == 0:
        left, right = -1, -1
    m = torch.ones(lq, lk, dtype=torch.bool)
    for i in range(lq):
        for j in range(lk):
            if left >= 0 and j < i + off - left:
                m[i, j] = False
            if right >= 0 and j > i + off + right:
                m[i, j] = False
    return m


@st.composite
def problems(draw):
    hkv = draw(st.integers(1, 2))
    hq = hkv * draw(st.integers(1, 3))
    mask = draw(st.integers(0, 3))
    nseg = draw(st.integers(1, 3))
    return dict(
        hq=hq, hkv=hkv, d=draw(st.sampled_from([4, 8])), dv=draw(st.sampled_from([3, 4, 8])), mask=mask,
        left=draw(st.integers(-1, 5)) if mask == 3 else -1, right=draw(st.integers(-1, 3)) if mask == 3 else -1,
        lq=[draw(st.integers(0, 9)) for _ in range(nseg)], lk=[draw(st.integers(0, 9)) for _ in range(nseg)],
        scale=draw(st.floats(0.1, 1.5)), seed=draw(st.integers(0, 2**31 - 1)))


@settings(max_examples=60, deadline=None)
@given(problems())
def test_oracle_equals_sdpa_per_segment(pb):
    F = torch.nn.functional
    g = torch.Generator().manual_seed(pb["seed"])
    tq, tk = sum(pb["lq"]), sum(pb["lk"])
    q = torch.randn(tq, pb["hq"], pb["d"], generator=g, dtype=F64)
    k = torch.randn(tk, pb["hkv"], pb["d"], generator=g, dtype=F64)
    v = torch.randn(tk, pb["hkv"], pb["dv"], generator=g, dtype=F64)
    do = torch.randn(tq, pb["hq"], pb["dv"], generator=g, dtype=F64)
    cu_q = torch.tensor([0] + list(torch.tensor(pb["lq"]).cumsum(0).tolist()), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(torch.tensor(pb["lk"]).cumsum(0).tolist()), dtype=torch.int32)
    kw = dict(mask=pb["mask"], left=pb["left"], right=pb["right"], cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    o, lse = R.attn_forward(q, k, v, pb["scale"], **kw)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, pb["scale"], **kw)
    dk_ref, dv_ref = torch.zeros_like(k), torch.zeros_like(v)
    for b, (lq, lk) in enumerate(zip(pb["lq"], pb["lk"])):
        rq = slice(int(cu_q[b]), int(cu_q[b + 1]))
        rk = slice(int(cu_k[b]), int(cu_k[b + 1]))
        if lq == 0:
            continue
        vis = mask_matrix(lq, lk, pb["mask"], pb["left"], pb["right"])
        live = vis.any(dim=1) if lk > 0 else torch.zeros(lq, dtype=torch.bool)
        dead = ~live
        # rows with no visible key: the oracle's reading
        assert (o[rq][dead] == 0).all() and (dq[rq][dead] == 0).all()
        assert torch.isinf(lse[:, rq][:, dead]).all() and (lse[:, rq][:, dead] < 0).all()
        if not bool(live.any()):
            continue
        qt = q[rq][live].permute(1, 0, 2).unsqueeze(0).clone().requires_grad_(True)
        kt = k[rk].permute(1, 0, 2).unsqueeze(0).clone().requires_grad_(True)
        vt = v[rk].permute(1, 0, 2).unsqueeze(0).clone().requires_grad_(True)
        ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=vis[live], scale=pb["scale"],
                                             enable_gqa=pb["hq"] != pb["hkv"])
        ref.backward(do[rq][live].permute(1, 0, 2).unsqueeze(0))
        tol = 1e-11
        assert torch.allclose(o[rq][live], ref.detach()[0].permute(1, 0, 2), atol=tol)
        assert torch.allclose(dq[rq][live], qt.grad[0].permute(1, 0, 2), atol=tol)
        dk_ref[rk] += kt.grad[0].permute(1, 0, 2)
        dv_ref[rk] += vt.grad[0].permute(1, 0, 2)
        # LSE: the log-sum-exp of the scaled visible scores, from the definition
        s = pb["scale"] * torch.einsum("ihd,jhd->hij", q[rq][live],
                                       k[rk].repeat_interleave(pb["hq"] // pb["hkv"], dim=1))
        s = s.masked_fill(~vis[live].unsqueeze(0), -math.inf)
        assert torch.allclose(lse[:, rq][:, live], torch.logsumexp(s, dim=2), atol=tol)
    assert torch.allclose(dk, dk_ref, atol=1e-11)
    assert torch.allclose(dv, dv_ref, atol=1e-11)
