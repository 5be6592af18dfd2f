"""GPU parity of the attention bias, dbias and dropout (through the C ABI)
against the fp64 oracle, element by element.

Bias shapes 11SS / 1HSS / BHSS / B1SS with dbias in BHSS, and dropout from
the philox seed / offset pair (TransformerEngine PR #446: the bias strides of
ck_fused_attn_bwd.cpp and the philox arguments of ck_attn_bwd).  The oracle
produces O and LSE with the same bias and dropout mask, rounded to the input
dtype, and both sides run the backward on those inputs; the dropout mask is
drawn on both sides from the same Philox4x32-10 counters, so dropped weights
agree exactly.  The CUDA-core forward helper's bias and dropout are checked
against the oracle's forward too.
"""
import numpy as np
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from oracle import attn_ref as R
from tests.parity import assert_all_ok, call_scale, compare, layout_heads_outer, per_segment_report, tolerances
from tests.test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

SHAPES = {"11SS": lambda b, h: (1, 1), "1HSS": lambda b, h: (1, h), "BHSS": lambda b, h: (b, h),
          "B1SS": lambda b, h: (b, 1)}


def _bias(kind, wl, seed):
    if kind is None:
        return None
    bb, bh = SHAPES[kind](wl.batch, wl.hq)
    g = torch.Generator().manual_seed(seed)
    return torch.randn((bb, bh, wl.sq, wl.sk), generator=g, dtype=torch.float32).to(wl.dtype)


def run_extras(B, wl, det, bias_kind=None, dropout_p=0.0, seed=0, offset=0, layout=None):
    """Oracle forward -> rounded O / fp32 LSE -> GPU and oracle backward with
    the same bias and dropout; reports per tensor, per segment and per
    (batch, head) slice of dbias."""
    x = wl.inputs()
    bias = _bias(bias_kind, wl, 7 + wl.seed)
    p32 = float(np.float32(dropout_p))     # the ABI takes the probability as fp32
    cu, cuk = wl.cu_seqlens(), wl.cu_seqlens_k()
    kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    okw = dict(kw, bias=bias, dropout_p=p32, philox_seed=seed, philox_offset=offset)
    o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **okw)
    o_in, lse_in = o64.to(wl.dtype), lse64.to(torch.float32)
    ref = R.attn_backward(x["q"], x["k"], x["v"], o_in, x["do"], lse_in, wl.scale,
                          return_dbias=bias is not None, **okw)
    dev = {k: v.cuda() for k, v in x.items()}
    dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    seed_t = torch.tensor([seed], dtype=torch.int64, device="cuda")
    off_t = torch.tensor([offset], dtype=torch.int64, device="cuda")
    out = tuple(torch.full_like(dev[n], float("nan")) for n in ("q", "k", "v"))
    dev["o"] = o_in.cuda()
    if layout is not None:   # strided views with the same values (the host may fold the batch into the heads)
        dev, out = layout(dev)
    got = B.attn_backward(dev["q"], dev["k"], dev["v"], dev["o"], dev["do"], lse_in.cuda(), scale=wl.scale,
                          deterministic=det, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, out=out,
                          bias=None if bias is None else bias.cuda(), return_dbias=bias is not None,
                          dropout_p=p32, philox_seed=seed_t, philox_offset=off_t, **dkw)
    torch.cuda.synchronize()
    tol, mcos = tolerances(wl.dtype)
    reps = []
    names = ("dq", "dk", "dv", "dbias")[:len(ref)]
    cf = call_scale(ref)
    for name, g, r in zip(names, got, ref):
        g = g.cpu()
        rep = compare(g, r, tol, mcos, cf)
        rep["tensor"] = name
        reps.append(rep)
        if name == "dbias":
            floor = max(float(r.abs().max()), cf)
            for b in range(r.shape[0]):
                for h in range(r.shape[1]):
                    rr = compare(g[b, h], r[b, h], tol, mcos, floor)
                    rr.update(tensor="dbias", batch=b, head=h)
                    reps.append(rr)
        elif cu is not None:
            offs = cu if name == "dq" else cuk
            reps.extend(per_segment_report(g, r, offs.tolist(), name, tol, mcos, call_floor=cf))
    return reps


def _wl(name, dtype, b, hq, hkv, sq, sk, d, dv, mask, left=-1, right=-1, seed=0):
    return W.Workload(name, dtype, b, hq, hkv, sq, sk, d, dv, mask, left, right, False, seed)


DET_MODES = dict(argvalues=[1, 2, 0], ids=["ordered", "split", "atomic"])
BASE = _wl("bias_causal", torch.bfloat16, 2, 4, 2, 200, 200, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=21)


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("kind", sorted(SHAPES))
def test_bias_shapes_and_dbias(B, kind, det):
    assert_all_ok(run_extras(B, BASE, det, bias_kind=kind), f"bias {kind} det={det}")


BIAS_MORE = [
    _wl("bias_window_fp16_d64", torch.float16, 1, 2, 2, 300, 300, 64, 64, W.MASK_WINDOW, 70, 5, seed=22),
    _wl("bias_nomask_sq_ne_sk", torch.bfloat16, 1, 2, 1, 150, 260, 128, 128, W.MASK_NONE, seed=23),
    _wl("bias_br_causal_d192", torch.bfloat16, 1, 2, 2, 140, 200, 192, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=24),
    _wl("bias_causal_d256", torch.bfloat16, 1, 2, 1, 180, 180, 256, 256, W.MASK_CAUSAL_TOP_LEFT, seed=25),
]


@pytest.mark.parametrize("det", [1, 0], ids=["det", "atomic"])
@pytest.mark.parametrize("wl", BIAS_MORE, ids=lambda w: w.name)
def test_bias_masks_and_head_dims(B, wl, det):
    assert_all_ok(run_extras(B, wl, det, bias_kind="BHSS"), f"{wl.name} det={det}")


@pytest.mark.parametrize("det", **DET_MODES)
def test_dropout(B, det):
    wl = _wl("drop_causal", torch.bfloat16, 2, 4, 2, 200, 200, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=31)
    assert_all_ok(run_extras(B, wl, det, dropout_p=0.25, seed=0x1234ABCD5678, offset=3), f"dropout det={det}")


def test_dropout_with_bias_fp16_window(B):
    wl = _wl("drop_bias", torch.float16, 1, 2, 1, 260, 260, 64, 64, W.MASK_WINDOW, 100, 0, seed=32)
    assert_all_ok(run_extras(B, wl, 1, bias_kind="1HSS", dropout_p=0.4, seed=99, offset=2**33 + 5),
                  "dropout with bias")


@pytest.mark.parametrize("det", [1, 0], ids=["det", "atomic"])
def test_dropout_packed_segments(B, det):
    wl = W.thd("drop_thd", [100, 80, 76], hq=8, hkv=2, seed=33)
    assert_all_ok(run_extras(B, wl, det, dropout_p=0.125, seed=7, offset=0), f"dropout THD det={det}")


@pytest.mark.parametrize("kind", ["1HSS", "B1SS", "BHSS"])
def test_bias_and_dropout_with_heads_outer_layout(B, kind):
    """Heads-outer tensors ([B, H, S, D] memory order): the host runs the call
    as one batch entry with B * H heads, so the kernel recovers the caller's
    (batch entry, head) for the bias and keeps b * Hq + h for the dropout
    counter and dbias."""
    assert_all_ok(run_extras(B, BASE, 1, bias_kind=kind, dropout_p=0.25, seed=77, offset=1,
                             layout=layout_heads_outer), f"heads-outer bias {kind}")


@pytest.mark.parametrize("kind,p", [("BHSS", 0.0), (None, 0.25), ("11SS", 0.3)])
def test_forward_helper_bias_and_dropout(B, kind, p):
    """The CUDA-core forward helper with bias and dropout against the oracle's
    forward (O and LSE)."""
    wl = _wl("fwd_extras", torch.bfloat16, 2, 4, 2, 150, 170, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=41)
    x = wl.inputs()
    bias = _bias(kind, wl, 9)
    p32 = float(np.float32(p))
    o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, mask=wl.mask, bias=bias, dropout_p=p32,
                                philox_seed=11, philox_offset=4)
    d = {k: v.cuda() for k, v in x.items()}
    o, lse = B.attn_forward(d["q"], d["k"], d["v"], scale=wl.scale, mask=wl.mask,
                            bias=None if bias is None else bias.cuda(), dropout_p=p32,
                            philox_seed=torch.tensor([11], dtype=torch.int64, device="cuda"),
                            philox_offset=torch.tensor([4], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    tol, mcos = tolerances(wl.dtype)
    assert compare(o.cpu(), o64, tol, mcos)["ok"]
    assert float((lse.cpu().double() - lse64).abs().max()) < 1e-3
