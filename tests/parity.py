"""Comparison helpers shared by the parity tests (no attention arithmetic).

Acceptance, per tensor and per packed segment: for 16-bit inputs, cosine
similarity >= 0.9999 and max|gpu - ref| <= 2e-2 * max|ref|; for fp32 inputs,
max|gpu - ref| <= 1e-4 * max|ref|.  Comparisons are made in fp64.
"""
from __future__ import annotations

import torch

BF16_TOL_REL = 2e-2
BF16_MIN_COS = 0.9999
FP32_TOL_REL = 1e-4


def tolerances(dtype):
    if dtype == torch.float32:
        return FP32_TOL_REL, 0.0
    return BF16_TOL_REL, BF16_MIN_COS


# A segment whose exact gradient is zero (every row sees a single key, so
# dS = P (dP - D) vanishes) still carries fp64 round-off in the oracle, of the
# order of 1e-16 of the tensor's scale.  Below this fraction of the tensor's
# max|ref| a segment counts as zero-signal.
ZERO_SIGNAL_REL = 1e-9


def call_scale(refs):
    """The largest max|ref| over the gradients of one call.  A whole tensor
    whose exact value is zero (with a single visible key per row, dQ and dK
    vanish while dV = sum of dO does not) is judged at this scale."""
    return max((float(r.detach().abs().max()) for r in refs if r.numel()), default=0.0)


def compare(got, ref, tol_rel, min_cos, scale_floor=0.0):
    """Max-abs-error and cosine check of one tensor (or one segment of it).

    Every tensor or segment with signal must satisfy, on its own scale,
    max|got - ref| <= tol_rel * max|ref| and (16-bit inputs) cosine >= min_cos.
    `scale_floor` is the max|ref| of the whole tensor when a segment is
    compared on its own, or the call's scale (`call_scale`) when a whole
    tensor is; it is used only for a zero-signal tensor or segment (its
    reference is at most ZERO_SIGNAL_REL * scale_floor, i.e. exactly zero up
    to fp64 round-off), whose bound is rounding noise at that scale because a
    fp32 kernel cannot reproduce an exact cancellation.
    """
    got = got.detach().to("cpu", torch.float64).reshape(-1)
    ref = ref.detach().to("cpu", torch.float64).reshape(-1)
    max_ref = float(ref.abs().max()) if ref.numel() else 0.0
    err = float((got - ref).abs().max()) if ref.numel() else 0.0
    finite = bool(torch.isfinite(got).all())
    ng, nr = float(got.norm()), float(ref.norm())
    if nr == 0.0 and ng == 0.0:
        cos = 1.0
    elif nr == 0.0 or ng == 0.0:
        cos = 0.0
    else:
        cos = float((got @ ref) / (ng * nr))
    zero_signal = max_ref <= ZERO_SIGNAL_REL * scale_floor
    if max_ref == 0.0 and scale_floor == 0.0:
        ok = finite and err == 0.0
    elif zero_signal:
        ok = finite and err <= tol_rel * scale_floor
    else:
        ok = finite and err <= tol_rel * max_ref and (min_cos <= 0.0 or cos >= min_cos)
    return dict(ok=ok, cos=cos, max_err=err, max_ref=max_ref, finite=finite, zero_signal=zero_signal)


def per_segment_report(got, ref, cu, name, tol_rel, min_cos, starts=None, call_floor=0.0):
    """One comparison per segment of a [T, H, D] tensor; segment b has length
    cu[b+1] - cu[b] and starts at row starts[b] (cu[b] when packed).  A
    zero-signal segment is judged at the tensor's scale, or at `call_floor`
    (the call's scale) when that is larger."""
    out = []
    cu = [int(x) for x in cu]
    starts = cu if starts is None else [int(x) for x in starts]
    floor = max(float(ref.detach().abs().max()) if ref.numel() else 0.0, call_floor)
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b]
        rows = slice(starts[b], starts[b] + n)
        r = compare(got[rows], ref[rows], tol_rel, min_cos, floor)
        r.update(tensor=name, segment=b, length=n)
        out.append(r)
    return out


def assert_all_ok(reports, what=""):
    bad = [r for r in reports if not r["ok"]]
    assert not bad, f"{what}: {len(bad)} failing comparisons, first: {bad[:3]}"


# Strided layouts (per-tensor {batch, row, head} strides).  Each layout turns
# contiguous device tensors into views with the same values and returns the
# output views (filled with NaN) that the gradients go to.
def _heads_outer(t):
    """The values of a [B,S,H,D] / [T,H,D] tensor in a [B,H,S,D] / [H,T,D] buffer."""
    if t.dim() == 4:
        return t.transpose(1, 2).contiguous().transpose(1, 2)
    return t.transpose(0, 1).contiguous().transpose(0, 1)


def layout_heads_outer(x):
    ins = {n: _heads_outer(t) for n, t in x.items()}
    outs = tuple(_heads_outer(torch.full_like(x[n], float("nan"))) for n in ("q", "k", "v"))
    return ins, outs


def _sbhd(t):
    """The values of a [B,S,H,D] tensor in an [S,B,H,D] buffer."""
    return t.transpose(0, 1).contiguous().transpose(0, 1)


def layout_sbhd(x):
    ins = {n: _sbhd(t) for n, t in x.items()}
    outs = tuple(_sbhd(torch.full_like(x[n], float("nan"))) for n in ("q", "k", "v"))
    return ins, outs


def layout_packed(x):
    """q, k, v (and dq, dk, dv) as slices of one [.., Hq + 2 Hkv, D] buffer per
    row (packed QKV; needs d_qk == d_v); o and dO with rows padded by 8."""
    hq, hkv = x["q"].shape[-2], x["k"].shape[-2]
    lead = x["q"].shape[:-2]

    def pack(q, k, v):
        buf = torch.full(lead + (hq + 2 * hkv, q.shape[-1]), float("nan"), dtype=q.dtype, device=q.device)
        buf[..., :hq, :], buf[..., hq:hq + hkv, :], buf[..., hq + hkv:, :] = q, k, v
        return buf[..., :hq, :], buf[..., hq:hq + hkv, :], buf[..., hq + hkv:, :]

    def pad_rows(t):
        buf = torch.full(lead + (t.shape[-2] + 1, t.shape[-1]), float("nan"), dtype=t.dtype, device=t.device)
        buf[..., :-1, :] = t
        return buf[..., :-1, :]

    q, k, v = pack(x["q"], x["k"], x["v"])
    ins = dict(q=q, k=k, v=v, o=pad_rows(x["o"]), do=pad_rows(x["do"]))
    nan = torch.full_like(x["q"], float("nan"))
    return ins, pack(nan, torch.full_like(x["k"], float("nan")), torch.full_like(x["v"], float("nan")))


STRIDED_LAYOUTS = (layout_heads_outer, layout_packed, layout_sbhd)
