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


def compare(got, ref, tol_rel, min_cos, scale_floor=0.0):
    """Max-abs-error and cosine check of one tensor (or one segment of it).

    `scale_floor` is the max|ref| of the whole tensor when a segment is
    compared on its own: the error bound is relative to the tensor's scale,
    so a segment whose reference is exactly zero (one visible key) accepts
    rounding noise at that scale instead of demanding exact zeros.
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
    bound = tol_rel * max(max_ref, scale_floor)
    ok = finite and err <= bound
    if max_ref > 0.0 and min_cos > 0.0:
        # cosine only where the segment has signal above the rounding floor
        if max_ref >= 10 * tol_rel * scale_floor:
            ok = ok and cos >= min_cos
    if max_ref == 0.0 and scale_floor == 0.0:
        ok = finite and err == 0.0
    return dict(ok=ok, cos=cos, max_err=err, max_ref=max_ref, finite=finite)


def per_segment_report(got, ref, cu, name, tol_rel, min_cos, starts=None):
    """One comparison per segment of a [T, H, D] tensor; segment b has length
    cu[b+1] - cu[b] and starts at row starts[b] (cu[b] when packed)."""
    out = []
    cu = [int(x) for x in cu]
    starts = cu if starts is None else [int(x) for x in starts]
    floor = float(ref.detach().abs().max()) if ref.numel() else 0.0
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
