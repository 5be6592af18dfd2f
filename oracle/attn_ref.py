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

Attention bias and dropout (TransformerEngine PR #446: the bias of shape
(bias_b, bias_h, s_q, s_kv) in the BiasShape kinds 11SS / 1HSS / BHSS / B1SS,
batch mode only, dbias returned in the BHSS shape; dropout driven by a philox
seed / offset pair passed to the backward):

8. The bias is added to the scaled scores before the mask:
   S = s Q K^T + bias[b', h'] with b' = b, h' = h on the dimensions the shape
   has and 0 on the broadcast ones; dbias[b, h] = dS (the gradient of the
   biased scores), in the full [B, Hq, Sq, Sk] shape.
9. Dropout keeps weight (i, j) of (batch or segment b, query head h) when a
   Philox4x32-10 word (Salmon, Moraes, Dror and Shaw, "Parallel random
   numbers: as easy as 1, 2, 3", SC'11) is at least floor(p * 2^32): key =
   (seed mod 2^32, seed div 2^32); counter = (lo32(n), j, b * Hq + h,
   hi32(n)) with n = offset + (i div 4); the word is number (i mod 4) of the
   four.  O = (P o Z / (1 - p)) V, LSE is that of P; in the backward
   dV = (P o Z / (1 - p))^T dO, dP = (dO V^T) o Z / (1 - p),
   dS = P o (dP - D) with D = rowsum(dO o O) as before.

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


# ---------------------------------------------------------------------------
# Philox counter-based generator, written from its published definition
# (Salmon et al., SC'11): N = 4 words of W bits, key of 2 words; each of the R
# rounds multiplies words 0 and 2 by M0 and M1 (full 2W-bit products), the
# outputs are (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
# lo(M0 c0)), and the key is bumped by the Weyl constants (W0, W1) between
# rounds.  The W = 64 instance is compared with numpy's Philox bit generator
# in the tests; the dropout mask uses W = 32.
# ---------------------------------------------------------------------------
PHILOX_CONSTANTS = {
    32: (0xD2511F53, 0xCD9E8D57, 0x9E3779B9, 0xBB67AE85),
    64: (0xD2E7470EE14C6C93, 0xCA5A826395121157, 0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B),
}


def philox(ctr, key, width=32, rounds=10):
    """Philox-4xW-R on Python ints or (for W = 32) numpy uint64 arrays holding
    W-bit values; returns the four output words."""
    m0, m1, w0, w1 = PHILOX_CONSTANTS[width]
    mask = (1 << width) - 1
    c0, c1, c2, c3 = ctr
    k0, k1 = key
    for r in range(rounds):
        if r > 0:
            k0, k1 = (k0 + w0) & mask, (k1 + w1) & mask
        p0, p1 = c0 * m0, c2 * m1          # W = 32: exact in uint64
        c0, c1, c2, c3 = (p1 >> width) ^ c1 ^ k0, p1 & mask, (p0 >> width) ^ c3 ^ k1, p0 & mask
    return c0, c1, c2, c3


def dropout_keep(lq: int, lk: int, bh: int, p: float, seed: int, offset: int) -> torch.Tensor:
    """Boolean [lq, lk] keep mask of one (batch or segment, query head) pair,
    bh = b * Hq + h (reading 9)."""
    import numpy as np
    u64 = np.uint64
    i = np.arange(lq, dtype=np.uint64).reshape(-1, 1)
    j = np.arange(lk, dtype=np.uint64).reshape(1, -1)
    n = (u64(offset) + (i >> u64(2))) & u64(0xFFFFFFFFFFFFFFFF)
    m32 = u64(0xFFFFFFFF)
    shape = (lq, lk)
    ctr = (np.broadcast_to(n & m32, shape).astype(np.uint64), np.broadcast_to(j, shape).astype(np.uint64),
           np.full(shape, bh, dtype=np.uint64), np.broadcast_to(n >> u64(32), shape).astype(np.uint64))
    key = (u64(seed & 0xFFFFFFFF), u64((seed >> 32) & 0xFFFFFFFF))
    words = np.stack(philox(ctr, key, 32), axis=0)            # [4, lq, lk]
    sel = np.broadcast_to((i & u64(3)).astype(np.int64), shape)
    r = np.take_along_axis(words, sel[None], axis=0)[0]
    thr = int(math.floor(p * 4294967296.0))
    return torch.from_numpy(r >= u64(thr))


def _bias_for(bias, b, h):
    """[Sq, Sk] bias of batch entry b, query head h (broadcast dims of size 1)."""
    return bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]


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


def _head_forward(qh, kh, vh, scale, vis, bias=None, keep=None, p_drop=0.0):
    """One head: S = s Q K^T (+ bias) masked, LSE, P, O = (P o Z / (1 - p)) V
    (all fp64); returns P before dropout."""
    s = scale * (qh @ kh.T)
    if bias is not None:
        s = s + bias
    s = s.masked_fill(~vis, -math.inf)
    m = s.max(dim=1, keepdim=True).values
    has = torch.isfinite(m)
    m0 = torch.where(has, m, torch.zeros_like(m))
    e = torch.exp(s - m0)
    lse = (torch.log(e.sum(dim=1, keepdim=True)) + m0).squeeze(1)
    lse = torch.where(has.squeeze(1), lse, torch.full_like(lse, -math.inf))
    p = _probs(s, lse)
    pv = p if keep is None else p * keep.to(F64) / (1.0 - p_drop)
    return p, lse, pv @ vh


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
                 cu_seqlens_k_padded=None, bias=None, dropout_p=0.0, philox_seed=0, philox_offset=0):
    """Forward pass: returns (O, LSE) in fp64 with the layouts of the header.
    `bias` ([bias_b, bias_h, Sq, Sk], batch mode) and dropout follow readings
    8 and 9."""
    batch_mode = cu_seqlens_q is None
    if bias is not None and not batch_mode:
        raise ValueError("the attention bias is defined for batch mode only")
    q, k, v = _as64(q), _as64(k), _as64(v)
    bias = None if bias is None else _as64(bias)
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
            keep = dropout_keep(lq, lk, b * hq + h, dropout_p, philox_seed, philox_offset) if dropout_p > 0 else None
            bias_h = None if bias is None else _bias_for(bias, b, h)
            _, lse_h, o_h = _head_forward(qb[:, h], kb[:, h // g], vb[:, h // g], scale, vis, bias_h, keep,
                                          dropout_p)
            if batch_mode:
                o[b, rq, h] = o_h
                lse[b, h, rq] = lse_h
            else:
                o[rq, h] = o_h
                lse[h, rq] = lse_h
    return o, lse


def attn_backward(q, k, v, o, do, lse, scale, mask=MASK_NONE, left=-1, right=-1,
                  cu_seqlens_q=None, cu_seqlens_k=None, cu_seqlens_q_padded=None,
                  cu_seqlens_k_padded=None, bias=None, dropout_p=0.0, philox_seed=0, philox_offset=0,
                  return_dbias=False):
    """Backward pass given the forward's O and LSE: returns (dQ, dK, dV) fp64,
    plus dbias [B, Hq, Sq, Sk] when return_dbias.

    Per (segment, query head h, kv head g = h // G):
      S = s Q K^T (+ bias) (masked -> -inf), P = exp(S - LSE),
      D_i = sum_c dO_ic O_ic, with F = Z / (1 - p) under dropout (else 1):
      dV_g += (P o F)^T dO, dP = (dO V^T) o F, dS = P o (dP - D),
      dQ = s dS K, dK_g += s dS^T Q, dbias = dS.
    """
    batch_mode = cu_seqlens_q is None
    if bias is not None and not batch_mode:
        raise ValueError("the attention bias is defined for batch mode only")
    q, k, v, o, do, lse = (_as64(t) for t in (q, k, v, o, do, lse))
    bias = None if bias is None else _as64(bias)
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    dbias = None
    if return_dbias:
        if not batch_mode:
            raise ValueError("dbias is defined for batch mode only")
        dbias = torch.zeros(q.shape[0], q.shape[2], q.shape[1], k.shape[1], dtype=F64)
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
            s = scale * (qh @ kh.T)
            if bias is not None:
                s = s + _bias_for(bias, b, h)
            s = s.masked_fill(~vis, -math.inf)
            p = _probs(s, lse_h)
            f = 1.0
            if dropout_p > 0:
                f = dropout_keep(lq, lk, b * hq + h, dropout_p, philox_seed, philox_offset).to(F64) / (1.0 - dropout_p)
            dvec = (doh * ob[:, h]).sum(dim=1)
            dvb[:, kvh] += (p * f).T @ doh
            dp = (doh @ vh.T) * f
            ds = p * (dp - dvec.view(-1, 1))
            dqb[:, h] = scale * (ds @ kh)
            dkb[:, kvh] += scale * (ds.T @ qh)
            if dbias is not None:
                dbias[b, h] = ds
    if return_dbias:
        return dq, dk, dv, dbias
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
