"""Pins for the fp64 oracle, independent of the oracle's own formulas.

Each check is chosen so that a plausible slip (dropped term, wrong sign,
transposed operand, wrong head mapping, wrong log base, wrong mask alignment)
fails at least one of them:

* central finite differences of L = sum(dO * O) w.r.t. Q, K, V;
* closed forms: one visible key; constant keys;
* exact invariants: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i over rows that see
  a key, sum <Q,dQ> = sum <K,dK>, dQ unchanged when every key is shifted;
* block-diagonal: a packed THD batch equals each segment alone
  (TransformerEngine PR #671, Verification);
* GQA: grouped dK/dV equal per-query-head gradients summed over the group;
* library routines: scipy's logsumexp, torch's scaled_dot_product_attention
  forward and its autograd backward;
* hand-written visibility matrices for the mask kinds (tests/golden).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def rnd(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64)


def loss(q, k, v, do, scale, **kw):
    o, _ = R.attn_forward(q, k, v, scale, **kw)
    return float((o * do).sum())


def fd_grad(x, f, h=1e-6):
    g = torch.zeros_like(x)
    flat, gflat = x.view(-1), g.view(-1)
    for i in range(flat.numel()):
        x0 = flat[i].item()
        flat[i] = x0 + h
        fp = f()
        flat[i] = x0 - h
        fm = f()
        flat[i] = x0
        gflat[i] = (fp - fm) / (2 * h)
    return g


def grads(q, k, v, do, scale, **kw):
    o, lse = R.attn_forward(q, k, v, scale, **kw)
    return R.attn_backward(q, k, v, o, do, lse, scale, **kw)


def rel_err(a, b):
    return float((a - b).abs().max() / max(b.abs().max().item(), 1e-9))


# ---------------------------------------------------------------- masks

def _read_masks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "mask_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) == 6:
                cur = dict(name=parts[0], lq=int(parts[1]), lk=int(parts[2]), mask=int(parts[3]),
                           left=int(parts[4]), right=int(parts[5]), rows=[])
                blocks.append(cur)
            else:
                cur["rows"].append([int(c) for c in parts[0]])
    return blocks


@pytest.mark.parametrize("blk", _read_masks(), ids=lambda b: b["name"])
def test_visibility_matches_hand_written(blk):
    got = R.visible(blk["lq"], blk["lk"], blk["mask"], blk["left"], blk["right"])
    assert got.int().tolist() == blk["rows"]


def test_visible_pairs_brute_force():
    for lq, lk, m, l, r in [(7, 7, 1, -1, 0), (5, 9, 2, -1, 0), (9, 5, 2, -1, 0), (10, 10, 3, 3, 0),
                            (10, 12, 3, 2, 1), (0, 4, 1, -1, 0)]:
        n = sum(1 for i in range(lq) for j in range(lk) if _brute_visible(i, j, lq, lk, m, l, r))
        assert R.visible_pairs(lq, lk, m, l, r) == n


def _brute_visible(i, j, lq, lk, m, l, r):
    if m == 0:
        return True
    off = 0 if m == 1 else lk - lq
    if m in (1, 2):
        l, r = -1, 0
    lo_ok = l < 0 or j >= i + off - l
    hi_ok = r < 0 or j <= i + off + r
    return lo_ok and hi_ok


# ------------------------------------------------------ finite differences

FD_CASES = [
    dict(name="nomask", B=1, sq=5, sk=5, hq=1, hkv=1, d=4, dv=4, kw=dict(mask=0)),
    dict(name="causal_tl", B=2, sq=5, sk=8, hq=2, hkv=2, d=4, dv=8, kw=dict(mask=1)),
    dict(name="causal_br_short_k", B=1, sq=8, sk=5, hq=2, hkv=1, d=8, dv=4, kw=dict(mask=2)),
    dict(name="window", B=1, sq=8, sk=8, hq=1, hkv=1, d=4, dv=4, kw=dict(mask=3, left=2, right=0)),
    dict(name="window_lr", B=1, sq=5, sk=8, hq=2, hkv=1, d=4, dv=4, kw=dict(mask=3, left=1, right=2)),
    dict(name="gqa", B=1, sq=5, sk=5, hq=4, hkv=2, d=4, dv=4, kw=dict(mask=1)),
    dict(name="one_row", B=1, sq=1, sk=1, hq=1, hkv=1, d=4, dv=4, kw=dict(mask=0)),
]


@pytest.mark.parametrize("c", FD_CASES, ids=lambda c: c["name"])
def test_finite_differences_batch(c):
    scale = 0.7
    q = rnd((c["B"], c["sq"], c["hq"], c["d"]), 1)
    k = rnd((c["B"], c["sk"], c["hkv"], c["d"]), 2)
    v = rnd((c["B"], c["sk"], c["hkv"], c["dv"]), 3)
    do = rnd((c["B"], c["sq"], c["hq"], c["dv"]), 4)
    dq, dk, dv = grads(q, k, v, do, scale, **c["kw"])
    f = lambda: loss(q, k, v, do, scale, **c["kw"])  # noqa: E731
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = fd_grad(x, f)
        assert rel_err(g, num) < 1e-6


def test_finite_differences_varlen():
    scale = 0.5
    cu = torch.tensor([0, 3, 8], dtype=torch.int32)
    q, k, v, do = rnd((8, 2, 4), 5), rnd((8, 1, 4), 6), rnd((8, 1, 4), 7), rnd((8, 2, 4), 8)
    kw = dict(mask=1, cu_seqlens_q=cu, cu_seqlens_k=cu)
    dq, dk, dv = grads(q, k, v, do, scale, **kw)
    f = lambda: loss(q, k, v, do, scale, **kw)  # noqa: E731
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert rel_err(g, fd_grad(x, f)) < 1e-6


def test_finite_differences_cross_attention_varlen():
    """Separate query and key offsets per segment, bottom-right causal: one
    segment with more keys than queries, one with fewer, one with no keys
    (its rows see nothing) and one with no queries."""
    scale = 0.6
    cu_q = torch.tensor([0, 3, 8, 10, 10], dtype=torch.int32)
    cu_k = torch.tensor([0, 6, 8, 8, 11], dtype=torch.int32)
    q, k, v, do = rnd((10, 2, 4), 9), rnd((11, 1, 4), 10), rnd((11, 1, 3), 11), rnd((10, 2, 3), 12)
    kw = dict(mask=2, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    dq, dk, dv = grads(q, k, v, do, scale, **kw)
    f = lambda: loss(q, k, v, do, scale, **kw)  # noqa: E731
    for x, g in ((q, dq), (k, dk), (v, dv)):
        assert rel_err(g, fd_grad(x, f)) < 1e-6
    assert (dq[8:10] == 0).all()          # segment with no keys
    assert (dk[8:11] == 0).all() and (dv[8:11] == 0).all()   # segment with no queries


def test_batch_problem_with_an_empty_side():
    """Batch layout with no keys at all: every row's softmax runs over nothing,
    so O = 0, LSE = -inf and dQ = 0 (the values of a fully masked row).  With
    no queries at all no key is seen: dK = dV = 0."""
    q, do = rnd((2, 5, 4, 6), 31), rnd((2, 5, 4, 3), 32)
    k0, v0 = rnd((2, 0, 2, 6), 33), rnd((2, 0, 2, 3), 34)
    o, lse = R.attn_forward(q, k0, v0, 0.4)
    assert o.shape == (2, 5, 4, 3) and (o == 0).all()
    assert lse.shape == (2, 4, 5) and torch.isneginf(lse).all()
    dq, dk, dv = R.attn_backward(q, k0, v0, o, do, lse, 0.4)
    assert (dq == 0).all() and dk.shape == k0.shape and dv.shape == v0.shape
    q0, k, v = rnd((2, 0, 4, 6), 35), rnd((2, 7, 2, 6), 36), rnd((2, 7, 2, 3), 37)
    for mask in (0, 1, 2):
        o, lse = R.attn_forward(q0, k, v, 0.4, mask=mask)
        dq, dk, dv = R.attn_backward(q0, k, v, o, torch.zeros_like(o), lse, 0.4, mask=mask)
        assert dq.shape == q0.shape and (dk == 0).all() and (dv == 0).all()


# ------------------------------------------------------------ closed forms

def test_single_key_closed_form():
    q, k, v, do = rnd((2, 6, 2, 4), 1), rnd((2, 1, 2, 4), 2), rnd((2, 1, 2, 3), 3), rnd((2, 6, 2, 3), 4)
    o, lse = R.attn_forward(q, k, v, 0.3)
    assert torch.allclose(o, v.expand(2, 6, 2, 3), atol=1e-14)
    expect_lse = (0.3 * (q * k).sum(-1)).permute(0, 2, 1)
    assert torch.allclose(lse, expect_lse, atol=1e-13)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.3)
    assert dq.abs().max() < 1e-13 and dk.abs().max() < 1e-13
    assert torch.allclose(dv, do.sum(dim=1, keepdim=True), atol=1e-13)


def test_constant_keys_uniform_probabilities():
    sq, sk = 6, 6
    q, v, do = rnd((1, sq, 1, 4), 1), rnd((1, sk, 1, 5), 2), rnd((1, sq, 1, 5), 3)
    k = rnd((1, 1, 1, 4), 4).expand(1, sk, 1, 4).clone()
    o, lse = R.attn_forward(q, k, v, 0.9, mask=1)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.9, mask=1)
    for i in range(sq):
        assert torch.allclose(o[0, i, 0], v[0, : i + 1, 0].mean(0), atol=1e-13)
    assert dq.abs().max() < 1e-12
    n_vis = torch.arange(1, sq + 1, dtype=F64)
    expect_dv = torch.stack([(do[0, j:, 0] / n_vis[j:].view(-1, 1)).sum(0) for j in range(sk)])
    assert torch.allclose(dv[0, :, 0], expect_dv, atol=1e-13)


# -------------------------------------------------------------- invariants

@pytest.mark.parametrize("mask,left,right,sq,sk", [(0, -1, -1, 9, 9), (1, -1, 0, 9, 12),
                                                   (2, -1, 0, 12, 7), (3, 3, 1, 10, 10)])
def test_exact_invariants(mask, left, right, sq, sk):
    B, hq, hkv, d, dv_ = 2, 4, 2, 8, 6
    q, k, v, do = (rnd((B, sq, hq, d), 11), rnd((B, sk, hkv, d), 12),
                   rnd((B, sk, hkv, dv_), 13), rnd((B, sq, hq, dv_), 14))
    kw = dict(mask=mask, left=left, right=right)
    o, lse = R.attn_forward(q, k, v, 0.4, **kw)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.4, **kw)
    vis = R.visible(sq, sk, mask, left, right)
    rows_alive = vis.any(dim=1)
    g = hq // hkv
    for b in range(B):
        for kvh in range(hkv):
            heads = list(range(kvh * g, (kvh + 1) * g))
            # sum_j dS_ij = 0  =>  sum_j dK_j = 0
            assert dk[b, :, kvh].sum(0).abs().max() < 1e-11
            # sum_j P_ij = 1 on live rows  =>  sum_j dV_j = sum_i dO_i (live rows)
            s_do = do[b][rows_alive][:, heads].sum(dim=(0, 1))
            assert torch.allclose(dv[b, :, kvh].sum(0), s_do, atol=1e-11)
            # bilinearity of Q K^T: sum <Q, dQ> = sum <K, dK>
            lhs = (q[b][:, heads] * dq[b][:, heads]).sum()
            rhs = (k[b, :, kvh] * dk[b, :, kvh]).sum()
            assert abs(float(lhs - rhs)) < 1e-11 * max(1.0, abs(float(lhs)))
    # shift invariance of softmax in the key direction: dQ unchanged
    c = rnd((1, 1, 1, d), 15)
    o2, lse2 = R.attn_forward(q, k + c, v, 0.4, **kw)
    dq2, _, _ = R.attn_backward(q, k + c, v, o2, do, lse2, 0.4, **kw)
    assert torch.allclose(dq, dq2, atol=1e-11)


def test_fully_masked_rows_are_zero():
    q, k, v, do = rnd((1, 6, 1, 4), 1), rnd((1, 3, 1, 4), 2), rnd((1, 3, 1, 4), 3), rnd((1, 6, 1, 4), 4)
    o, lse = R.attn_forward(q, k, v, 1.0, mask=2)
    dead = ~R.visible(6, 3, 2).any(dim=1)
    assert dead.sum() == 3
    assert torch.isinf(lse[0, 0, dead]).all() and (lse[0, 0, dead] < 0).all()
    assert (o[0, dead] == 0).all()
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 1.0, mask=2)
    assert (dq[0, dead] == 0).all()
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()


# ------------------------------------------------------ structural invariants

def test_block_diagonal_packed_equals_segments():
    segs = [5, 1, 9, 3]
    cu = torch.tensor(np.cumsum([0] + segs), dtype=torch.int32)
    t = sum(segs)
    q, k, v, do = rnd((t, 4, 8), 21), rnd((t, 2, 8), 22), rnd((t, 2, 6), 23), rnd((t, 4, 6), 24)
    kw = dict(mask=3, left=2, right=0)
    o, lse = R.attn_forward(q, k, v, 0.35, cu_seqlens_q=cu, cu_seqlens_k=cu, **kw)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.35, cu_seqlens_q=cu, cu_seqlens_k=cu, **kw)
    for b in range(len(segs)):
        r = slice(int(cu[b]), int(cu[b + 1]))
        ob, lseb = R.attn_forward(q[r][None], k[r][None], v[r][None], 0.35, **kw)
        assert torch.allclose(o[r], ob[0], atol=1e-13)
        assert torch.allclose(lse[:, r], lseb[0], atol=1e-13)
        g = R.attn_backward(q[r][None], k[r][None], v[r][None], ob, do[r][None], lseb, 0.35, **kw)
        for packed, alone in zip((dq, dk, dv), g):
            assert torch.allclose(packed[r], alone[0], atol=1e-13)


def test_block_diagonal_cross_attention_equals_segments():
    """Packed segments with their own key lengths equal batch-mode attention of
    each segment alone (Sq = its query length, Sk = its key length); a segment
    with no keys has LSE = -inf and O = dQ = 0."""
    lq, lk = [4, 7, 0, 3, 5], [9, 2, 4, 0, 5]
    cu_q = torch.tensor(np.cumsum([0] + lq), dtype=torch.int32)
    cu_k = torch.tensor(np.cumsum([0] + lk), dtype=torch.int32)
    tq, tk = sum(lq), sum(lk)
    q, k, v, do = rnd((tq, 4, 8), 25), rnd((tk, 2, 8), 26), rnd((tk, 2, 6), 27), rnd((tq, 4, 6), 28)
    for kw in (dict(mask=2), dict(mask=1), dict(mask=3, left=2, right=1), dict(mask=0)):
        seg = dict(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
        o, lse = R.attn_forward(q, k, v, 0.35, **seg, **kw)
        dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.35, **seg, **kw)
        for b in range(len(lq)):
            rq = slice(int(cu_q[b]), int(cu_q[b + 1]))
            rk = slice(int(cu_k[b]), int(cu_k[b + 1]))
            if lk[b] == 0:
                assert torch.isinf(lse[:, rq]).all() and (lse[:, rq] < 0).all()
                assert (o[rq] == 0).all() and (dq[rq] == 0).all()
                continue
            if lq[b] == 0:
                assert (dk[rk] == 0).all() and (dv[rk] == 0).all()
                continue
            ob, lseb = R.attn_forward(q[rq][None], k[rk][None], v[rk][None], 0.35, **kw)
            assert torch.allclose(o[rq], ob[0], atol=1e-13)
            assert torch.equal(torch.isinf(lse[:, rq]), torch.isinf(lseb[0]))
            fin = torch.isfinite(lseb[0])
            assert torch.allclose(lse[:, rq][fin], lseb[0][fin], atol=1e-13)
            g = R.attn_backward(q[rq][None], k[rk][None], v[rk][None], ob, do[rq][None], lseb, 0.35, **kw)
            for packed, alone, r in zip((dq, dk, dv), g, (rq, rk, rk)):
                assert torch.allclose(packed[r], alone[0], atol=1e-13)


def test_padded_layout_equals_packed():
    """A padded THD layout (segment starts from the padded offsets, lengths from
    cu_seqlens) gives, on the segments' rows, exactly the packed result of the
    same segments; rows of no segment get zero gradients, O = 0, LSE = -inf.
    Padding rows hold large garbage so that any leak shows."""
    lq, lk = [4, 7, 0, 3, 5], [9, 2, 4, 0, 5]
    gq, gk = [1, 2, 0, 3, 1, 2], [0, 3, 1, 2, 0, 4]
    cu_q = torch.tensor(np.cumsum([0] + lq), dtype=torch.int32)
    cu_k = torch.tensor(np.cumsum([0] + lk), dtype=torch.int32)

    def starts(lens, gaps):
        st, r = [], 0
        for b, n in enumerate(lens):
            r += gaps[b]
            st.append(r)
            r += n
        return torch.tensor(st + [r + gaps[-1]], dtype=torch.int32)

    st_q, st_k = starts(lq, gq), starts(lk, gk)
    tq, tk = int(st_q[-1]), int(st_k[-1])
    q, k, v, do = rnd((sum(lq), 4, 8), 41), rnd((sum(lk), 2, 8), 42), rnd((sum(lk), 2, 6), 43), rnd((sum(lq), 4, 6), 44)

    def spread(x, cu, st, total, seed):
        out = 1e3 * rnd((total,) + tuple(x.shape[1:]), seed)
        for b in range(len(cu) - 1):
            n = int(cu[b + 1] - cu[b])
            out[int(st[b]):int(st[b]) + n] = x[int(cu[b]):int(cu[b + 1])]
        return out

    def gather(x, cu, st):
        return torch.cat([x[int(st[b]):int(st[b]) + int(cu[b + 1] - cu[b])] for b in range(len(cu) - 1)])

    qp, dop = spread(q, cu_q, st_q, tq, 45), spread(do, cu_q, st_q, tq, 46)
    kp, vp = spread(k, cu_k, st_k, tk, 47), spread(v, cu_k, st_k, tk, 48)
    pad_q = torch.ones(tq, dtype=torch.bool)
    pad_q[torch.cat([torch.arange(int(st_q[b]), int(st_q[b]) + lq[b]) for b in range(5)])] = False
    pad_k = torch.ones(tk, dtype=torch.bool)
    pad_k[torch.cat([torch.arange(int(st_k[b]), int(st_k[b]) + lk[b]) for b in range(5)])] = False
    for kw in (dict(mask=2), dict(mask=3, left=2, right=1), dict(mask=0)):
        packed = dict(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, **kw)
        padded = dict(cu_seqlens_q_padded=st_q, cu_seqlens_k_padded=st_k, **packed)
        o, lse = R.attn_forward(q, k, v, 0.4, **packed)
        grads_packed = R.attn_backward(q, k, v, o, do, lse, 0.4, **packed)
        op, lsep = R.attn_forward(qp, kp, vp, 0.4, **padded)
        assert torch.equal(gather(op, cu_q, st_q), o)
        assert torch.equal(gather(lsep.T, cu_q, st_q), lse.T)
        assert (op[pad_q] == 0).all() and torch.isneginf(lsep[:, pad_q]).all()
        opg = spread(o, cu_q, st_q, tq, 49)          # garbage O and LSE in padding rows
        lsepg = spread(lse.T, cu_q, st_q, tq, 50).T
        dq, dk, dv = R.attn_backward(qp, kp, vp, opg, dop, lsepg, 0.4, **padded)
        assert torch.equal(gather(dq, cu_q, st_q), grads_packed[0])
        assert torch.equal(gather(dk, cu_k, st_k), grads_packed[1])
        assert torch.equal(gather(dv, cu_k, st_k), grads_packed[2])
        assert (dq[pad_q] == 0).all() and (dk[pad_k] == 0).all() and (dv[pad_k] == 0).all()


def test_gqa_equals_summed_mha():
    B, s, hq, hkv, d = 1, 7, 6, 2, 4
    q, k, v, do = rnd((B, s, hq, d), 31), rnd((B, s, hkv, d), 32), rnd((B, s, hkv, d), 33), rnd((B, s, hq, d), 34)
    dq, dk, dv = grads(q, k, v, do, 0.5, mask=1)
    g = hq // hkv
    kr, vr = k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2)
    dq_m, dk_m, dv_m = grads(q, kr, vr, do, 0.5, mask=1)
    assert torch.allclose(dq, dq_m, atol=1e-13)
    assert torch.allclose(dk, dk_m.view(B, s, hkv, g, d).sum(3), atol=1e-13)
    assert torch.allclose(dv, dv_m.view(B, s, hkv, g, d).sum(3), atol=1e-13)


# ---------------------------------------------------------- library routines

def test_lse_matches_scipy_logsumexp():
    scipy_special = pytest.importorskip("scipy.special")
    q, k, v = rnd((1, 9, 2, 8), 41), rnd((1, 11, 2, 8), 42), rnd((1, 11, 2, 8), 43)
    _, lse = R.attn_forward(q, k, v, 0.25, mask=3, left=4, right=1)
    vis = R.visible(9, 11, 3, 4, 1).numpy()
    for h in range(2):
        s = 0.25 * (q[0, :, h].numpy() @ k[0, :, h].numpy().T)
        s = np.where(vis, s, -np.inf)
        np.testing.assert_allclose(lse[0, h].numpy(), scipy_special.logsumexp(s, axis=1), rtol=0, atol=1e-13)


@pytest.mark.parametrize("mask,sq,sk,hq,hkv", [(0, 6, 9, 2, 2), (1, 9, 9, 4, 2), (2, 6, 9, 2, 1),
                                              (3, 10, 10, 2, 2)])
def test_matches_torch_sdpa_and_autograd(mask, sq, sk, hq, hkv):
    F = torch.nn.functional
    B, d, dv_ = 2, 8, 5
    left, right = (3, 1) if mask == 3 else (-1, -1)
    q, k, v, do = rnd((B, sq, hq, d), 51), rnd((B, sk, hkv, d), 52), rnd((B, sk, hkv, dv_), 53), rnd((B, sq, hq, dv_), 54)
    vis = R.visible(sq, sk, mask, left, right)
    qt, kt, vt = (x.permute(0, 2, 1, 3).clone().requires_grad_(True) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=vis, scale=0.45, enable_gqa=hkv != hq)
    ref.backward(do.permute(0, 2, 1, 3))
    o, lse = R.attn_forward(q, k, v, 0.45, mask=mask, left=left, right=right)
    assert torch.allclose(o, ref.detach().permute(0, 2, 1, 3), atol=1e-12)
    dq, dk, dv = R.attn_backward(q, k, v, o, do, lse, 0.45, mask=mask, left=left, right=right)
    assert torch.allclose(dq, qt.grad.permute(0, 2, 1, 3), atol=1e-12)
    assert torch.allclose(dk, kt.grad.permute(0, 2, 1, 3), atol=1e-12)
    assert torch.allclose(dv, vt.grad.permute(0, 2, 1, 3), atol=1e-12)


# ------------------------------------------------------ sampled-row helpers

def test_sampled_rows_match_full_backward():
    segs = [40, 1, 70]
    cu = torch.tensor(np.cumsum([0] + segs), dtype=torch.int32)
    t = sum(segs)
    q, k, v, do = rnd((t, 4, 8), 61), rnd((t, 2, 8), 62), rnd((t, 2, 8), 63), rnd((t, 4, 8), 64)
    kw = dict(mask=1, cu_seqlens_q=cu, cu_seqlens_k=cu)
    dq, dk, dv = grads(q, k, v, do, 0.3, **kw)
    for b in range(3):
        n = segs[b]
        rows = [0, n - 1, n // 2]
        for h in range(4):
            got = R.dq_rows(q, k, v, do, 0.3, b, h, rows, **kw)
            assert torch.allclose(got, dq[int(cu[b]) + torch.tensor(rows), h], atol=1e-13)
        for kvh in range(2):
            gk, gv = R.dkv_rows(q, k, v, do, 0.3, b, kvh, rows, **kw)
            assert torch.allclose(gk, dk[int(cu[b]) + torch.tensor(rows), kvh], atol=1e-13)
            assert torch.allclose(gv, dv[int(cu[b]) + torch.tensor(rows), kvh], atol=1e-13)


def test_sampled_rows_batch_window():
    B, s = 2, 33
    q, k, v, do = rnd((B, s, 2, 8), 71), rnd((B, s, 1, 8), 72), rnd((B, s, 1, 4), 73), rnd((B, s, 2, 4), 74)
    kw = dict(mask=3, left=5, right=0)
    dq, dk, dv = grads(q, k, v, do, 0.3, **kw)
    rows = [0, 7, 32]
    gk, gv = R.dkv_rows(q, k, v, do, 0.3, 1, 0, rows, **kw)
    assert torch.allclose(gk, dk[1, rows, 0], atol=1e-13) and torch.allclose(gv, dv[1, rows, 0], atol=1e-13)
    assert torch.allclose(R.dq_rows(q, k, v, do, 0.3, 1, 1, rows, **kw), dq[1, rows, 1], atol=1e-13)


# ------------------------------------------------------- planted mistakes
# Each plants a plausible slip into the oracle's inputs or a copy of its
# result on the CPU and checks that one of the pins above rejects it.

def _fd_rel_err(grad_fn):
    q, k, v, do = rnd((1, 5, 1, 4), 81), rnd((1, 5, 1, 4), 82), rnd((1, 5, 1, 4), 83), rnd((1, 5, 1, 4), 84)
    dq, dk, dv = grad_fn(q, k, v, do)
    f = lambda: loss(q, k, v, do, 0.6, mask=1)  # noqa: E731
    return max(rel_err(dq, fd_grad(q, f)), rel_err(dk, fd_grad(k, f)), rel_err(dv, fd_grad(v, f)))


def test_planted_dropped_d_term_is_caught():
    def bad(q, k, v, do):
        o, lse = R.attn_forward(q, k, v, 0.6, mask=1)
        return R.attn_backward(q, k, v, torch.zeros_like(o), do, lse, 0.6, mask=1)
    assert _fd_rel_err(bad) > 1e-2


def test_planted_log2_lse_is_caught():
    def bad(q, k, v, do):
        o, lse = R.attn_forward(q, k, v, 0.6, mask=1)
        return R.attn_backward(q, k, v, o, do, lse / math.log(2.0), 0.6, mask=1)
    assert _fd_rel_err(bad) > 1e-2


def test_planted_transposed_mask_is_caught():
    def bad(q, k, v, do):
        o, lse = R.attn_forward(q, k, v, 0.6, mask=1)
        # the backward evaluated with the opposite triangle
        return R.attn_backward(q.flip(1), k.flip(1), v.flip(1), o.flip(1), do.flip(1), lse.flip(2), 0.6, mask=1)
    assert _fd_rel_err(bad) > 1e-2


def test_page3_failure_signature_is_detected():
    """The THD bug of PR #671: every segment past offset 0 lands on the
    offset-0 slot, so only segment 0 of dQ is right.  The per-segment check
    used by the GPU tests must flag exactly the later segments."""
    from tests.parity import per_segment_report
    page = json.load(open(os.path.join(GOLDEN, "page3_verification.json")))
    segs = page["splits"][1]
    cu = np.cumsum([0] + segs)
    t = int(cu[-1])
    cu_t = torch.tensor(cu, dtype=torch.int32)
    q, k, v, do = rnd((t, 2, 8), 91), rnd((t, 1, 8), 92), rnd((t, 1, 8), 93), rnd((t, 2, 8), 94)
    dq, _, _ = grads(q, k, v, do, 0.3, mask=1, cu_seqlens_q=cu_t, cu_seqlens_k=cu_t)
    broken = dq.clone()
    for b in range(1, len(segs)):
        n = segs[b]
        broken[int(cu[b]): int(cu[b]) + n] = rnd((n, 2, 8), 95 + b)  # never written: garbage
    rep = per_segment_report(broken, dq, cu, "dq", tol_rel=2e-2, min_cos=0.9999)
    assert [r["ok"] for r in rep] == [True, False, False]
    rep_good = per_segment_report(dq, dq, cu, "dq", tol_rel=2e-2, min_cos=0.9999)
    assert all(r["ok"] for r in rep_good)
