"""Plain fp64 CPU oracle for the fused multi-head attention (FMHA) backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (no kernels, headers, helpers or constants).

What it computes is the textbook softmax-attention forward and backward, in
float64 on the CPU, one (batch or segment, query head) at a time, with dense
score matrices and library matmuls as the only primitives.  Sources:

* ROCm/aiter PR #2216 "[CK_TILE] FMHA BWD Use Persistent Kernels in
  Deterministic Mode", Motivation: the backward produces dQ/dK/dV; dQ is
  accumulated in split fp32 slices and converted back.  The split workspace is
  an implementation device only, so the oracle has none.
* ROCm/TransformerEngine PR #671 "[ROCm] Fix THD/ragged dQ backward ...",
  Summary / Verification: packed THD (ragged) attention is checked against a
  block-diagonal reference, i.e. every segment attends only to itself.
* ROCm/TransformerEngine PR #446 "Update AITER subcommit ...", review of
  ``ck_to_aiter_mask_type``: mask kinds are "no mask", causal aligned top-left
  (1), causal aligned bottom-right (2) and a generic left/right window (3).

Readings where the pages are silent:

1. Visibility of key j to query i, with off = 0 (top-left) or Lk - Lq
   (bottom-right):  causal  <=>  j <= i + off;  window(left, right)  <=>
   i + off - left <= j <= i + off + right, inclusive, -1 meaning unbounded on
   that side.  The window kind is aligned bottom-right (off = Lk - Lq), the
   FlashAttention convention; with Lq == Lk both alignments coincide.
2. A row with no visible key has LSE = -inf, P = 0, O = 0 and zero gradients.
3. LSE is the natural-log log-sum-exp of the scaled scores.
4. The softmax scale s multiplies the raw scores; dQ and dK carry the factor
   s, dS does not.
5. GQA: query head h reads kv head h // (Hq / Hkv) (contiguous groups).
6. Group (THD) mode: segment b owns query rows cu_q[b]:cu_q[b+1] and key rows
   cu_k[b]:cu_k[b+1]; the result is the block-diagonal one.
7. Padded group mode (TransformerEngine PR #446, review of
   ck_fused_attn_fwd.cpp / ck_fused_attn_bwd.cpp: the segment start comes
   from the padded offsets when they are given, the length from cu_seqlens):
   segment b owns rows st[b] : st[b] + (cu[b+1] - cu[b]).  Rows of no segment
   get zero gradients, O = 0 and LSE = -inf.

Layouts (the same as the C ABI): batch mode q [B,Sq,Hq,d], k [B,Sk,Hkv,d],
v [B,Sk,Hkv,dv], o/do [B,Sq,Hq,dv], lse [B,Hq,Sq]; group mode drops B and
uses the packed token axis: q [Tq,Hq,d], lse [Hq,Tq].

Pins (tests/test_oracle.py): central finite differences, closed forms
(one visible key, constant keys), the exact invariants sum_j dS_ij = 0,
sum dV = sum dO, <Q,dQ> = <K,dK>, the block-diagonal and GQA invariants,
torch's own scaled_dot_product_attention (forward and autograd backward) and
scipy's logsumexp.
"""
from __future__ import annotations

import math

import torch

MASK_NONE = 0
MASK_CAUSAL_TOP_LEFT = 1
MASK_CAUSAL_BOTTOM_RIGHT = 2
MASK_WINDOW = 3

F64 = torch.float64


def _as64(x):
    return x.detach().to(device="cpu", dtype=F64)


def visible(lq: int, lk: int, mask: int, left: int = -1, right: int = -1) -> torch.Tensor:
    """Boolean [lq, lk] matrix: True where query i may attend to key j.

    Mask kinds follow the AITER mask enum reviewed in TransformerEngine PR #446
    (``ck_to_aiter_mask_type``); the predicates are reading 1 of the header.
    """
    i = torch.arange(lq).view(-1, 1)
    j = torch.arange(lk).view(1, -1)
    if mask == MASK_NONE:
        return torch.ones(lq, lk, dtype=torch.bool)
    if mask == MASK_CAUSAL_TOP_LEFT:
        off, left, right = 0, -1, 0
    elif mask == MASK_CAUSAL_BOTTOM_RIGHT:
        off, left, right = lk - lq, -1, 0
    elif mask == MASK_WINDOW:
        off = lk - lq
    else:
        raise ValueError(f"unknown mask kind {mask}")
    ok = torch.ones(lq, lk, dtype=torch.bool)
    if left >= 0:
        ok &= j >= i + off - left
    if right >= 0:
        ok &= j <= i + off + right
    return ok


def _rows(cu, st, b):
    """Physical rows of segment b: start st[b] (cu[b] when unpadded), length
    cu[b+1] - cu[b] (reading 7)."""
    n = int(cu[b + 1]) - int(cu[b])
    r0 = int(cu[b]) if st is None else int(st[b])
    return slice(r0, r0 + n)


def _segments(batch_mode: bool, nseg: int, sq: int, sk: int, cu_q, cu_k, st_q=None, st_k=None):
    """(query slice, key slice) per batch entry or packed segment."""
    out = []
    for b in range(nseg):
        if batch_mode:
            out.append((b, slice(0, sq), slice(0, sk)))
        else:
            out.append((b, _rows(cu_q, st_q, b), _rows(cu_k, st_k, b)))
    return out


def _views(x, batch_mode, b, rows):
    """[rows, H, dim] view of one batch entry / segment."""
    return x[b, rows] if batch_mode else x[rows]


def _head_forward(qh, kh, vh, scale, vis):
    """One head: S = s Q K^T masked, LSE, P, O (all fp64)."""
    s = scale * (qh @ kh.T)
    s = s.masked_fill(~vis, -math.inf)
    m = s.max(dim=1, keepdim=True).values
    has = torch.isfinite(m)
    m0 = torch.where(has, m, torch.zeros_like(m))
    e = torch.exp(s - m0)
    lse = (torch.log(e.sum(dim=1, keepdim=True)) + m0).squeeze(1)
    lse = torch.where(has.squeeze(1), lse, torch.full_like(lse, -math.inf))
    p = _probs(s, lse)
    return p, lse, p @ vh


def _probs(s, lse):
    """P = exp(S - LSE); rows with LSE = -inf (nothing visible) are zero."""
    dead = torch.isinf(lse) & (lse < 0)
    lse0 = torch.where(dead, torch.zeros_like(lse), lse)
    p = torch.exp(s - lse0.view(-1, 1))
    p = torch.where(torch.isfinite(s), p, torch.zeros_like(p))
    p[dead] = 0.0
    return p


def attn_forward(q, k, v, scale, mask=MASK_NONE, left=-1, right=-1,
                 cu_seqlens_q=None, cu_seqlens_k=None, cu_seqlens_q_padded=None,
                 cu_seqlens_k_padded=None):
    """Forward pass: returns (O, LSE) in fp64 with the layouts of the header."""
    batch_mode = cu_seqlens_q is None
    q, k, v = _as64(q), _as64(k), _as64(v)
    if batch_mode:
        nseg, sq, hq = q.shape[0], q.shape[1], q.shape[2]
        sk, hkv = k.shape[1], k.shape[2]
        o = torch.zeros(q.shape[:3] + (v.shape[-1],), dtype=F64)
        lse = torch.full((nseg, hq, sq), -math.inf, dtype=F64)
    else:
        nseg, sq, sk = len(cu_seqlens_q) - 1, None, None
        hq, hkv = q.shape[1], k.shape[1]
        o = torch.zeros(q.shape[:2] + (v.shape[-1],), dtype=F64)
        lse = torch.full((hq, q.shape[0]), -math.inf, dtype=F64)
    g = hq // hkv
    for b, rq, rk in _segments(batch_mode, nseg, sq, sk, cu_seqlens_q, cu_seqlens_k,
                               cu_seqlens_q_padded, cu_seqlens_k_padded):
        qb, kb, vb = _views(q, batch_mode, b, rq), _views(k, batch_mode, b, rk), _views(v, batch_mode, b, rk)
        lq, lk = qb.shape[0], kb.shape[0]
        if lq == 0 or lk == 0:   # no keys: every row keeps LSE = -inf and O = 0 (reading 2)
            continue
        vis = visible(lq, lk, mask, left, right)
        for h in range(hq):
            _, lse_h, o_h = _head_forward(qb[:, h], kb[:, h // g], vb[:, h // g], scale, vis)
            if batch_mode:
                o[b, rq, h] = o_h
                lse[b, h, rq] = lse_h
            else:
                o[rq, h] = o_h
                lse[h, rq] = lse_h
    return o, lse


def attn_backward(q, k, v, o, do, lse, scale, mask=MASK_NONE, left=-1, right=-1,
                  cu_seqlens_q=None, cu_seqlens_k=None, cu_seqlens_q_padded=None,
                  cu_seqlens_k_padded=None):
    """Backward pass given the forward's O and LSE: returns (dQ, dK, dV) fp64.

    Per (segment, query head h, kv head g = h // G):
      S = s Q K^T (masked -> -inf), P = exp(S - LSE), D_i = sum_c dO_ic O_ic,
      dV_g += P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = s dS K,
      dK_g += s dS^T Q.
    """
    batch_mode = cu_seqlens_q is None
    q, k, v, o, do, lse = (_as64(t) for t in (q, k, v, o, do, lse))
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    if batch_mode:
        nseg, sq, hq, sk, hkv = q.shape[0], q.shape[1], q.shape[2], k.shape[1], k.shape[2]
    else:
        nseg, sq, sk, hq, hkv = len(cu_seqlens_q) - 1, None, None, q.shape[1], k.shape[1]
    g = hq // hkv
    for b, rq, rk in _segments(batch_mode, nseg, sq, sk, cu_seqlens_q, cu_seqlens_k,
                               cu_seqlens_q_padded, cu_seqlens_k_padded):
        qb, kb, vb = _views(q, batch_mode, b, rq), _views(k, batch_mode, b, rk), _views(v, batch_mode, b, rk)
        ob, dob = _views(o, batch_mode, b, rq), _views(do, batch_mode, b, rq)
        dqb, dkb, dvb = _views(dq, batch_mode, b, rq), _views(dk, batch_mode, b, rk), _views(dv, batch_mode, b, rk)
        lq, lk = qb.shape[0], kb.shape[0]
        if lq == 0 or lk == 0:
            continue
        vis = visible(lq, lk, mask, left, right)
        for h in range(hq):
            kvh = h // g
            lse_h = lse[b, h, rq] if batch_mode else lse[h, rq]
            qh, kh, vh, doh = qb[:, h], kb[:, kvh], vb[:, kvh], dob[:, h]
            s = (scale * (qh @ kh.T)).masked_fill(~vis, -math.inf)
            p = _probs(s, lse_h)
            dvec = (doh * ob[:, h]).sum(dim=1)
            dvb[:, kvh] += p.T @ doh
            dp = doh @ vh.T
            ds = p * (dp - dvec.view(-1, 1))
            dqb[:, h] = scale * (ds @ kh)
            dkb[:, kvh] += scale * (ds.T @ qh)
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Sampled outputs for full-size workloads: each value is computed from
# Q, K, V and dO alone (no O or LSE taken from anywhere else).
# ---------------------------------------------------------------------------

def _segment_tensors(q, k, v, do, b, cu_q, cu_k):
    if cu_q is None:
        return q[b], k[b], v[b], do[b], 0, 0
    q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
    return q[q0:q1], k[k0:k1], v[k0:k1], do[q0:q1], q0, k0


def dq_rows(q, k, v, do, scale, b, h, rows, mask=MASK_NONE, left=-1, right=-1,
            cu_seqlens_q=None, cu_seqlens_k=None):
    """dQ[rows, h, :] of batch entry / segment b (rows are segment-local).

    Recomputes, for just these query rows, S = s q K^T, LSE, P, O = P V,
    D = rowsum(dO o O), dP = dO V^T, dS and dQ = s dS K, in fp64.
    """
    qs, ks, vs, dos, _, _ = _segment_tensors(q, k, v, do, b, cu_seqlens_q, cu_seqlens_k)
    hkv = ks.shape[1]
    g = qs.shape[1] // hkv
    rows = torch.as_tensor(rows, dtype=torch.long)
    qh, kh, vh, doh = _as64(qs[rows, h]), _as64(ks[:, h // g]), _as64(vs[:, h // g]), _as64(dos[rows, h])
    vis = visible(qs.shape[0], ks.shape[0], mask, left, right)[rows]
    p, _, oh = _head_forward(qh, kh, vh, scale, vis)
    dvec = (doh * oh).sum(dim=1)
    ds = p * (doh @ vh.T - dvec.view(-1, 1))
    return scale * (ds @ kh)


def dkv_rows(q, k, v, do, scale, b, hkv_idx, key_rows, mask=MASK_NONE, left=-1, right=-1,
             cu_seqlens_q=None, cu_seqlens_k=None):
    """(dK, dV)[key_rows, hkv_idx, :] of batch entry / segment b.

    Needs LSE and D of every query of the group's heads, so each head's full
    forward is recomputed here in fp64; the gradients are then formed only for
    the requested key columns and summed over the query heads of the group.
    """
    qs, ks, vs, dos, _, _ = _segment_tensors(q, k, v, do, b, cu_seqlens_q, cu_seqlens_k)
    hq, hkv = qs.shape[1], ks.shape[1]
    g = hq // hkv
    key_rows = torch.as_tensor(key_rows, dtype=torch.long)
    kh, vh = _as64(ks[:, hkv_idx]), _as64(vs[:, hkv_idx])
    vis = visible(qs.shape[0], ks.shape[0], mask, left, right)
    dk = torch.zeros(len(key_rows), kh.shape[1], dtype=F64)
    dv = torch.zeros(len(key_rows), vh.shape[1], dtype=F64)
    for h in range(hkv_idx * g, (hkv_idx + 1) * g):
        qh, doh = _as64(qs[:, h]), _as64(dos[:, h])
        p, _, oh = _head_forward(qh, kh, vh, scale, vis)
        dvec = (doh * oh).sum(dim=1)
        pc = p[:, key_rows]
        dv += pc.T @ doh
        dsc = pc * (doh @ vh[key_rows].T - dvec.view(-1, 1))
        dk += scale * (dsc.T @ qh)
    return dk, dv


def visible_pairs(lq: int, lk: int, mask: int, left: int = -1, right: int = -1) -> int:
    """Number of visible (query, key) pairs of one head of one segment."""
    if lq == 0 or lk == 0:
        return 0
    return int(visible(lq, lk, mask, left, right).sum())
