"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every element; they span several KV and query tiles with
ragged tails.  Packed THD cases are compared segment by segment (the failure
mode of TransformerEngine PR #671: first segment right, later ones garbage).
Full-size workloads are checked on sampled rows the oracle recomputes from
Q, K, V and dO alone (tests/test_gpu_fullsize.py).
"""
import math

import numpy as np
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from oracle import attn_ref as R
from tests.parity import (STRIDED_LAYOUTS, assert_all_ok, call_scale, compare, layout_heads_outer,
                          layout_packed, layout_sbhd, per_segment_report, tolerances)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_backward_gb300 import build, binding
    build.build_library()
    binding.load()
    return binding


def _wl(name, dtype, b, hq, hkv, s_q, s_k, dqk, dv, mask, left=-1, right=-1, seed=0, seqlens=None):
    return W.Workload(name, dtype, b, hq, hkv, s_q, s_k, dqk, dv, mask, left, right, False, seed,
                      seqlens)


def run_backward_vs_oracle(B, wl, deterministic, ref_fwd=True):
    """Oracle forward -> rounded O / fp32 LSE -> GPU backward and oracle backward
    on identical inputs; returns reports per tensor (and per segment)."""
    x = wl.inputs()
    cu, cuk = wl.cu_seqlens(), wl.cu_seqlens_k()
    stq, stk = wl.cu_seqlens_q_padded(), wl.cu_seqlens_k_padded()
    kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    if stq is not None or stk is not None:
        kw.update(cu_seqlens_q_padded=stq, cu_seqlens_k_padded=stk)
    o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **kw)
    o_in, lse_in = o64.to(wl.dtype), lse64.to(torch.float32)
    ref = R.attn_backward(x["q"], x["k"], x["v"], o_in, x["do"], lse_in, wl.scale, **kw)
    dev = {k: v.cuda() for k, v in x.items()}
    dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    # outputs start as NaN: every row, padding included, must be written
    out = tuple(torch.full_like(dev[n], float("nan")) for n in ("q", "k", "v"))
    got = B.attn_backward(dev["q"], dev["k"], dev["v"], o_in.cuda(), dev["do"], lse_in.cuda(),
                          scale=wl.scale, deterministic=deterministic, max_seqlen_q=wl.sq,
                          max_seqlen_k=wl.sk, out=out, **dkw)
    torch.cuda.synchronize()
    tol, mcos = tolerances(wl.dtype)
    cf = call_scale(ref)
    reps = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.cpu()
        rep = compare(g, r, tol, mcos, cf)
        rep["tensor"] = name
        reps.append(rep)
        if cu is not None:
            offs, st = (cu, stq) if name == "dq" else (cuk, stk)
            reps.extend(per_segment_report(g, r, offs.tolist(), name, tol, mcos,
                                           None if st is None else st.tolist(), call_floor=cf))
            pad = wl.padding_rows("q" if name == "dq" else "k")
            if pad:
                zero = bool((g[pad] == 0).all())
                reps.append(dict(ok=zero, tensor=name, padding_rows=len(pad), all_zero=zero))
    return reps


SMALL = [
    _wl("fp32_tiny", torch.float32, 1, 2, 2, 64, 64, 32, 32, W.MASK_NONE, seed=0),
    _wl("fp32_causal_ragged", torch.float32, 2, 2, 1, 150, 150, 64, 64, W.MASK_CAUSAL_TOP_LEFT, seed=1),
    _wl("bf16_causal_ragged", torch.bfloat16, 2, 2, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=2),
    _wl("bf16_gqa_causal", torch.bfloat16, 1, 4, 2, 257, 257, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=3),
    _wl("bf16_nomask_sq_ne_sk", torch.bfloat16, 1, 2, 1, 200, 333, 128, 128, W.MASK_NONE, seed=4),
    _wl("bf16_causal_br_long_k", torch.bfloat16, 1, 2, 2, 100, 300, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=5),
    _wl("bf16_causal_br_short_k", torch.bfloat16, 1, 2, 2, 300, 100, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=6),
    _wl("bf16_causal_tl_long_k", torch.bfloat16, 1, 2, 2, 100, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=7),
    _wl("bf16_window_left", torch.bfloat16, 1, 2, 2, 520, 520, 128, 128, W.MASK_WINDOW, 100, 0, seed=8),
    _wl("bf16_window_lr", torch.bfloat16, 1, 2, 1, 300, 350, 128, 128, W.MASK_WINDOW, 30, 20, seed=9),
    _wl("bf16_d64_causal", torch.bfloat16, 2, 2, 1, 200, 200, 64, 64, W.MASK_CAUSAL_TOP_LEFT, seed=10),
    _wl("bf16_d192_window", torch.bfloat16, 1, 2, 2, 400, 400, 192, 128, W.MASK_WINDOW, 150, 0, seed=11),
    _wl("fp16_causal", torch.float16, 1, 2, 2, 200, 200, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=12),
    _wl("bf16_d256_causal_ragged", torch.bfloat16, 2, 4, 2, 300, 300, 256, 256, W.MASK_CAUSAL_TOP_LEFT, seed=13),
    _wl("fp16_d256_window_sq_ne_sk", torch.float16, 1, 2, 1, 200, 333, 256, 256, W.MASK_WINDOW, 90, 10, seed=14),
    _wl("bf16_d256_nomask_one_tile", torch.bfloat16, 1, 2, 2, 64, 128, 256, 256, W.MASK_NONE, seed=15),
    # a single key: dQ and dK are exactly zero (dS = P (dP - D) cancels), dV = sum of dO
    _wl("bf16_single_key", torch.bfloat16, 2, 4, 2, 150, 1, 128, 128, W.MASK_NONE, seed=16),
    _wl("fp32_single_key", torch.float32, 1, 2, 1, 70, 1, 32, 32, W.MASK_NONE, seed=17),
    _wl("fp16_d192_single_key_window", torch.float16, 1, 2, 2, 90, 1, 192, 128, W.MASK_WINDOW, 5, 0, seed=18),
]


DET_MODES = dict(argvalues=[1, 2, 0], ids=["ordered", "split", "atomic"])


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_small_backward(B, wl, det):
    assert_all_ok(run_backward_vs_oracle(B, wl, det), wl.name)


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("heads", [(8, 2), (32, 8)], ids=["hq8_hkv2", "hq32_hkv8"])
@pytest.mark.parametrize("segs", W.PAGE_SPLITS + [[1, 1, 130, 1], [5, 0, 7], [2048]], ids=str)
def test_thd_splits_per_segment(B, segs, heads, det):
    """Packed THD, padding-causal within segments, GQA heads: a small group and
    the Llama-3-8B shape of the packed benchmark workload (32 query, 8 kv
    heads); every segment of every tensor is compared on its own
    (TransformerEngine PR #671, Tests / Verification)."""
    hq, hkv = heads
    wl = W.thd("thd", segs, hq=hq, hkv=hkv, seed=sum(segs) + hq)
    reps = run_backward_vs_oracle(B, wl, det)
    assert_all_ok(reps, f"segments {segs}")


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_thd_head_dim_256_per_segment(B, dtype, det):
    """Packed THD at head dim 256: each KV tile's two column-half passes are
    work items of their own, and in the ordered fold each half has its own
    turn counters; every segment is compared with the oracle."""
    wl = W.thd("thd_d256", [300, 1, 129, 200, 64], hq=4, hkv=2, d_qk=256, d_v=256, dtype=dtype, seed=47)
    assert_all_ok(run_backward_vs_oracle(B, wl, det), "thd d256")


# Cross-attention varlen: every segment has its own query and key length,
# including segments with no keys (their dQ is zero) and no queries (their
# dK, dV are zero), lengths off the 128-row tile and segments longer than one
# KV tile on one side only.
ASYM_Q = [100, 0, 37, 250, 5, 129, 300]
ASYM_K = [300, 64, 0, 129, 200, 128, 17]


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("mask,left,right", [(W.MASK_NONE, -1, -1),
                                             (W.MASK_CAUSAL_BOTTOM_RIGHT, -1, -1),
                                             (W.MASK_CAUSAL_TOP_LEFT, -1, -1),
                                             (W.MASK_WINDOW, 40, 8)],
                         ids=["nomask", "causal_br", "causal_tl", "window"])
def test_thd_cross_attention_lengths(B, mask, left, right, det):
    """Separate query and key offsets per packed segment (cu_seqlens_q differs
    from cu_seqlens_k), compared per segment on each side."""
    wl = W.thd("thd_cross", ASYM_Q, hq=4, hkv=2, mask=mask, left=left, right=right,
               seed=101 + mask, seqlens_k=ASYM_K)
    assert_all_ok(run_backward_vs_oracle(B, wl, det), f"cross-attention varlen mask {mask}")


# Padded THD: segment rows start at the padded offsets, lengths come from
# cu_seqlens; gaps before the first segment, between segments (longer than a
# tile, and zero) and after the last one, on either side alone or both.
PAD_Q = [100, 0, 37, 250, 5, 129]
PAD_K = [300, 64, 0, 129, 200, 128]
PADDED = [
    dict(name="both", gaps_q=[3, 0, 17, 1, 140, 2, 9], gaps_k=[0, 5, 0, 131, 7, 1, 30]),
    dict(name="q_only", gaps_q=[0, 1, 2, 3, 4, 5, 6], gaps_k=None),
    dict(name="k_only", gaps_q=None, gaps_k=[8, 0, 0, 0, 0, 0, 0]),
]


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("pad", PADDED, ids=lambda c: c["name"])
@pytest.mark.parametrize("mask", [W.MASK_CAUSAL_BOTTOM_RIGHT, W.MASK_NONE], ids=["causal_br", "nomask"])
def test_thd_padded_layout(B, pad, mask, det):
    """cu_seqlens_q_padded / cu_seqlens_k_padded (TransformerEngine PR #446,
    review of ck_fused_attn_bwd.cpp): per-segment parity on the physical rows
    and exact zeros in every padding row of dQ, dK, dV."""
    wl = W.thd("thd_padded", PAD_Q, hq=4, hkv=2, mask=mask, seed=131 + mask, seqlens_k=PAD_K,
               gaps_q=pad["gaps_q"], gaps_k=pad["gaps_k"])
    assert_all_ok(run_backward_vs_oracle(B, wl, det), f"padded THD {pad['name']} mask {mask}")


def test_thd_padded_fp32(B):
    wl = W.thd("thd_padded_fp32", [70, 5, 130], hq=2, hkv=1, d_qk=64, d_v=64, dtype=torch.float32,
               seed=141, gaps_q=[2, 3, 0, 4], gaps_k=[0, 1, 64, 3])
    assert_all_ok(run_backward_vs_oracle(B, wl, 1), "padded THD fp32")


def run_strided_vs_oracle(B, wl, det, layout):
    x = wl.inputs()
    cu, cuk = wl.cu_seqlens(), wl.cu_seqlens_k()
    stq, stk = wl.cu_seqlens_q_padded(), wl.cu_seqlens_k_padded()
    kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    if stq is not None or stk is not None:
        kw.update(cu_seqlens_q_padded=stq, cu_seqlens_k_padded=stk)
    o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **kw)
    o_in, lse_in = o64.to(wl.dtype), lse64.to(torch.float32)
    ref = R.attn_backward(x["q"], x["k"], x["v"], o_in, x["do"], lse_in, wl.scale, **kw)
    dev = {n: t.cuda() for n, t in dict(x, o=o_in).items()}
    ins, out = layout(dev)
    assert not ins["q"].is_contiguous() and not out[0].is_contiguous()
    dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    got = B.attn_backward(ins["q"], ins["k"], ins["v"], ins["o"], ins["do"], lse_in.cuda(), scale=wl.scale,
                          deterministic=det, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, out=out, **dkw)
    torch.cuda.synchronize()
    tol, mcos = tolerances(wl.dtype)
    cf = call_scale(ref)
    reps = []
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.cpu()
        rep = compare(g, r, tol, mcos, cf)
        rep["tensor"] = name
        reps.append(rep)
        if cu is not None:
            offs, st = (cu, stq) if name == "dq" else (cuk, stk)
            reps.extend(per_segment_report(g, r, offs.tolist(), name, tol, mcos,
                                           None if st is None else st.tolist(), call_floor=cf))
    return reps


STRIDED = [
    (_wl("bf16_gqa_causal_ragged", torch.bfloat16, 2, 4, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=51),
     layout_heads_outer),
    (_wl("bf16_mha_window", torch.bfloat16, 2, 2, 2, 257, 257, 128, 128, W.MASK_WINDOW, 40, 0, seed=52),
     layout_packed),
    (_wl("bf16_d192_br_long_k", torch.bfloat16, 1, 2, 1, 100, 300, 192, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=53),
     layout_heads_outer),
    (_wl("bf16_d64_gqa", torch.bfloat16, 2, 4, 1, 200, 200, 64, 64, W.MASK_CAUSAL_TOP_LEFT, seed=54),
     layout_packed),
    (W.thd("thd_gqa", [100, 0, 37, 250, 5], hq=4, hkv=2, seed=55), layout_packed),
    (W.thd("thd_cross_padded", [100, 0, 37, 250], hq=4, hkv=2, mask=W.MASK_CAUSAL_BOTTOM_RIGHT, seed=56,
           seqlens_k=[300, 64, 0, 129], gaps_q=[3, 0, 17, 140, 2], gaps_k=[0, 5, 131, 7, 1]), layout_heads_outer),
    (_wl("fp32_causal", torch.float32, 2, 2, 1, 150, 150, 64, 64, W.MASK_CAUSAL_TOP_LEFT, seed=57),
     layout_heads_outer),
    (_wl("bf16_gqa_nomask_sq_ne_sk", torch.bfloat16, 3, 4, 2, 200, 333, 128, 128, W.MASK_NONE, seed=58),
     layout_sbhd),
    (_wl("fp16_window_lr", torch.float16, 2, 2, 1, 300, 350, 128, 128, W.MASK_WINDOW, 30, 20, seed=59),
     layout_sbhd),
]


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("case", STRIDED, ids=lambda c: f"{c[0].name}-{c[1].__name__[7:]}")
def test_strided_layouts(B, case, det):
    """Non-contiguous q/k/v/o/dO and dq/dk/dv (heads-outer buffers, packed QKV
    slices, padded rows) give the oracle's gradients; every output element is
    written (outputs start as NaN)."""
    wl, layout = case
    assert_all_ok(run_strided_vs_oracle(B, wl, det, layout), f"{wl.name} {layout.__name__}")


def test_forward_negative_scale_takes_cuda_core_path(B):
    """The tensor-core forward takes the row max on raw scores and needs a
    positive scale; a negative one runs the CUDA-core forward, still exact."""
    wl = SMALL[2]
    x = wl.inputs()
    o_ref, lse_ref = R.attn_forward(x["q"], x["k"], x["v"], -0.05, mask=wl.mask)
    o, lse = B.attn_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), scale=-0.05, mask=wl.mask)
    torch.cuda.synchronize()
    tol, mcos = tolerances(wl.dtype)
    assert compare(o.cpu(), o_ref, tol, mcos)["ok"]
    fin = torch.isfinite(lse_ref)
    assert float((lse.cpu().double()[fin] - lse_ref[fin]).abs().max()) < 1e-3


def test_forward_helper_strided(B):
    for wl, layout in STRIDED[:2] + STRIDED[4:6]:
        x = wl.inputs()
        kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=wl.cu_seqlens(),
                  cu_seqlens_k=wl.cu_seqlens_k())
        if wl.gaps_q or wl.gaps_k:
            kw.update(cu_seqlens_q_padded=wl.cu_seqlens_q_padded(), cu_seqlens_k_padded=wl.cu_seqlens_k_padded())
        o_ref, lse_ref = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **kw)
        dev = {n: t.cuda() for n, t in x.items()}
        dev["o"] = torch.zeros(x["do"].shape, dtype=wl.dtype, device="cuda")
        ins, _ = layout(dev)
        dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
        o, lse = B.attn_forward(ins["q"], ins["k"], ins["v"], scale=wl.scale, max_seqlen_q=wl.sq,
                                max_seqlen_k=wl.sk, **dkw)
        torch.cuda.synchronize()
        tol, mcos = tolerances(wl.dtype)
        assert compare(o.cpu(), o_ref, tol, mcos)["ok"], wl.name
        fin = torch.isfinite(lse_ref)
        assert torch.equal(torch.isfinite(lse.cpu()), fin)
        assert float((lse.cpu().double()[fin] - lse_ref[fin]).abs().max()) < 1e-3


def test_thd_window_and_d192(B):
    wl = W.thd("thd_win", [100, 300, 37], hq=4, hkv=4, d_qk=192, d_v=128, mask=W.MASK_WINDOW,
               left=64, right=0, seed=77)
    assert_all_ok(run_backward_vs_oracle(B, wl, True), "thd window d192")


def test_forward_helper_matches_oracle(B):
    cross = W.thd("t_cross_padded", PAD_Q, hq=4, hkv=2, mask=W.MASK_CAUSAL_BOTTOM_RIGHT, seed=4,
                  seqlens_k=PAD_K, gaps_q=PADDED[0]["gaps_q"], gaps_k=PADDED[0]["gaps_k"])
    # SMALL[0] (fp32) runs the CUDA-core forward, the 16-bit cases the tensor-core one
    for wl in (SMALL[0], SMALL[2], SMALL[3], SMALL[4], SMALL[6], SMALL[8], SMALL[9], SMALL[10], SMALL[11], SMALL[12],
               W.thd("t", [100, 80, 76], hq=4, hkv=2, seed=3), cross):
        x = wl.inputs()
        kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=wl.cu_seqlens(),
                  cu_seqlens_k=wl.cu_seqlens_k())
        if wl.gaps_q or wl.gaps_k:
            kw.update(cu_seqlens_q_padded=wl.cu_seqlens_q_padded(), cu_seqlens_k_padded=wl.cu_seqlens_k_padded())
        o_ref, lse_ref = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **kw)
        dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
        o, lse = B.attn_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), scale=wl.scale,
                                max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, **dkw)
        torch.cuda.synchronize()
        tol, mcos = tolerances(wl.dtype)
        assert compare(o.cpu(), o_ref, tol, mcos)["ok"], wl.name
        fin = torch.isfinite(lse_ref)
        assert torch.equal(torch.isfinite(lse.cpu()), fin)
        assert float((lse.cpu().double()[fin] - lse_ref[fin]).abs().max()) < 1e-3


def test_fully_masked_rows_give_zero_and_finite(B):
    wl = _wl("br_dead_rows", torch.bfloat16, 1, 2, 2, 300, 100, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=21)
    x = wl.inputs()
    o, lse = B.attn_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), scale=wl.scale, mask=wl.mask)
    dq, dk, dv = B.attn_backward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), o, x["do"].cuda(), lse,
                                 scale=wl.scale, mask=wl.mask, deterministic=True)
    torch.cuda.synchronize()
    dead = ~R.visible(300, 100, wl.mask).any(dim=1)
    assert int(dead.sum()) == 200
    assert torch.isinf(lse.cpu()[0, :, dead]).all()
    assert (dq.cpu()[0, dead] == 0).all()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


def test_gpu_forward_then_backward_end_to_end(B):
    """GPU forward -> GPU backward against the oracle's forward+backward."""
    wl = _wl("e2e", torch.bfloat16, 2, 4, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=31)
    x = wl.inputs()
    d = {k: v.cuda() for k, v in x.items()}
    o, lse = B.attn_forward(d["q"], d["k"], d["v"], scale=wl.scale, mask=wl.mask)
    got = B.attn_backward(d["q"], d["k"], d["v"], o, d["do"], lse, scale=wl.scale, mask=wl.mask,
                          deterministic=True)
    o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, mask=wl.mask)
    ref = R.attn_backward(x["q"], x["k"], x["v"], o64, x["do"], lse64, wl.scale, mask=wl.mask)
    reps = [compare(g.cpu(), r, 2e-2, 0.9999) for g, r in zip(got, ref)]
    assert_all_ok(reps, "e2e")


def _bwd_runs(B, wl, modes, repeats):
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    cu = wl.cu_seqlens()
    cu_d = None if cu is None else cu.cuda()
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu_d,
              cu_seqlens_k=cu_d, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o, lse = B.attn_forward(x["q"], x["k"], x["v"], **kw)
    out = {}
    for m in modes:
        out[m] = [[t.clone() for t in B.attn_backward(x["q"], x["k"], x["v"], o, x["do"], lse,
                                                       deterministic=m, **kw)] for _ in range(repeats)]
    return out


DET_CASES = [
    _wl("det_rep", torch.bfloat16, 2, 8, 2, 1000, 1000, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=41),
    _wl("det_win192", torch.bfloat16, 1, 4, 2, 700, 700, 192, 128, W.MASK_WINDOW, 200, 0, seed=42),
    _wl("det_br_short_k", torch.bfloat16, 1, 4, 4, 500, 300, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, seed=43),
    W.thd("det_thd", [700, 1, 129, 300, 64], hq=8, hkv=2, seed=44),
    # head dim 256: two column-half passes per KV tile, each with its own turn counters
    _wl("det_d256", torch.bfloat16, 1, 4, 2, 600, 600, 256, 256, W.MASK_CAUSAL_TOP_LEFT, seed=45),
    W.thd("det_thd_d256", [300, 1, 129, 200], hq=4, hkv=2, d_qk=256, d_v=256, seed=46),
]


@pytest.mark.parametrize("wl", DET_CASES, ids=lambda w: w.name)
def test_deterministic_bitwise_repeatable(B, wl):
    """Both deterministic modes give the same bits on 10 runs, and the ordered
    fold gives the same bits as the split slices (same additions, same order)."""
    runs = _bwd_runs(B, wl, (B.DET_ORDERED, B.DET_SPLIT), 10)
    for m, rs in runs.items():
        for again in rs[1:]:
            for a, b in zip(rs[0], again):
                assert torch.equal(a, b), f"mode {m} not repeatable"
    for a, b in zip(runs[B.DET_ORDERED][0], runs[B.DET_SPLIT][0]):
        assert torch.equal(a, b), "ordered fold differs from split slices"


@pytest.mark.parametrize("wl", [DET_CASES[0], DET_CASES[2], DET_CASES[3], DET_CASES[5]], ids=lambda w: w.name)
def test_ordered_fold_ignores_workspace_contents(B, wl):
    """The ordered fold initialises what it reads: its dQ slice, the turn
    counters and the tables (det_br_short_k has query tiles no KV tile reaches,
    whose dQ rows are zero).  A workspace filled with NaN bytes gives the same
    bits as a zeroed one."""
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    cu = wl.cu_seqlens()
    cu_d = None if cu is None else cu.cuda()
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu_d,
              cu_seqlens_k=cu_d, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o, lse = B.attn_forward(x["q"], x["k"], x["v"], **kw)
    res = []
    for fill in (0, 0xFF):
        outs = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]))
        p = B.bwd_params(x["q"], x["k"], x["v"], o, x["do"], lse, *outs, deterministic=B.DET_ORDERED, **kw)
        n = B.workspace_bytes(p)
        ws = B.alloc_workspace(n, x["q"].device)
        ws.fill_(fill)
        s = torch.cuda.current_stream().cuda_stream
        assert B.attn_bwd(p, ws.data_ptr(), n, s) == 0
        st, dev = B.attn_bwd_read_status(ws.data_ptr(), s)
        assert st == 0 and dev == 0
        res.append(outs)
    for a, b in zip(*res):
        assert not torch.isnan(b.float()).any()
        assert torch.equal(a, b)


@pytest.mark.parametrize("det", **DET_MODES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("sq,sk", [(0, 200), (200, 0), (0, 0)], ids=["no_queries", "no_keys", "neither"])
def test_batch_problem_with_an_empty_side(B, sq, sk, dtype, det):
    """No keys at all: the forward gives O = 0 and LSE = -inf (a fully masked
    row's values) and the backward dQ = 0; no queries at all: dK = dV = 0.  The
    outputs start as NaN, so every row must be written; the status is ok even
    after a failed call on the same workspace."""
    g = torch.Generator().manual_seed(sq + sk)
    rnd = lambda *shape: torch.randn(*shape, generator=g).to(dtype).cuda()  # noqa: E731
    d = 64 if dtype == torch.float32 else 128   # head dims of each dtype's backward
    q, k, v = rnd(2, sq, 4, d), rnd(2, sk, 2, d), rnd(2, sk, 2, d)
    do = rnd(2, sq, 4, d)
    o, lse = B.attn_forward(q, k, v, scale=0.088, mask=W.MASK_CAUSAL_BOTTOM_RIGHT)
    if sk == 0:
        assert (o == 0).all() and torch.isneginf(lse).all()
    ws = B.alloc_workspace(16 << 20, q.device)   # above the size these problems need
    ws[:4].copy_(torch.tensor([-6], dtype=torch.int32).view(torch.uint8))   # a stale failure status
    out = tuple(torch.full_like(t, float("nan")) for t in (q, k, v))
    dq, dk, dv = B.attn_backward(q, k, v, o, do, lse, scale=0.088, mask=W.MASK_CAUSAL_BOTTOM_RIGHT,
                                 deterministic=det, out=out, workspace=ws)
    torch.cuda.synchronize()
    if sk == 0:
        assert (dq == 0).all()
    if sq == 0:
        assert (dk == 0).all() and (dv == 0).all()


@pytest.mark.parametrize("det", **DET_MODES)
def test_packed_problem_without_keys(B, det):
    """Packed THD whose key side is empty in every segment: dQ = 0 for every
    row, the forward's O = 0 and LSE = -inf."""
    cu_q = torch.tensor([0, 100, 100, 163], dtype=torch.int32, device="cuda")
    cu_k = torch.zeros(4, dtype=torch.int32, device="cuda")
    q = torch.randn(163, 4, 128, device="cuda").to(torch.bfloat16)
    k = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    kw = dict(scale=0.088, mask=W.MASK_CAUSAL_BOTTOM_RIGHT, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
              max_seqlen_q=100, max_seqlen_k=0)
    o, lse = B.attn_forward(q, k, k, **kw)
    assert (o == 0).all() and torch.isneginf(lse).all()
    out = (torch.full_like(q, float("nan")), torch.empty_like(k), torch.empty_like(k))
    dq, _, _ = B.attn_backward(q, k, k, o, torch.randn_like(q), lse, deterministic=det, out=out, **kw)
    torch.cuda.synchronize()
    assert (dq == 0).all()


def test_bad_cu_seqlens_reported_by_device(B):
    wl = W.thd("bad", [100, 80, 76], hq=4, hkv=2)
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    bad = torch.tensor([0, 100, 90, 256], dtype=torch.int32, device="cuda")   # not monotone
    lse = torch.zeros(4, 256, device="cuda")
    with pytest.raises(B.AttnError) as e:
        B.attn_backward(x["q"], x["k"], x["v"], x["do"], x["do"], lse, scale=wl.scale, mask=1,
                        cu_seqlens_q=bad, cu_seqlens_k=bad, max_seqlen_q=100, max_seqlen_k=100)
    assert e.value.status == -7
    too_long = torch.tensor([0, 200, 230, 256], dtype=torch.int32, device="cuda")  # 200 > declared 100
    with pytest.raises(B.AttnError) as e:
        B.attn_backward(x["q"], x["k"], x["v"], x["do"], x["do"], lse, scale=wl.scale, mask=1,
                        cu_seqlens_q=too_long, cu_seqlens_k=too_long, max_seqlen_q=100, max_seqlen_k=100)
    assert e.value.status == -7
    # padded starts that overlap a segment, run past the rows, or start before row 0
    cu = torch.tensor([0, 100, 180, 256], dtype=torch.int32, device="cuda")
    for starts in ([0, 90, 190, 256], [0, 100, 180, 300], [-4, 100, 180, 256], [0, 100, 181, 256]):
        st = torch.tensor(starts, dtype=torch.int32, device="cuda")
        for side in ("cu_seqlens_q_padded", "cu_seqlens_k_padded"):
            out = tuple(torch.full_like(t, 7.0) for t in (x["q"], x["k"], x["v"]))
            with pytest.raises(B.AttnError) as e:
                B.attn_backward(x["q"], x["k"], x["v"], x["do"], x["do"], lse, scale=wl.scale, mask=1,
                                cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=100, max_seqlen_k=100,
                                out=out, **{side: st})
            assert e.value.status == -7, (starts, side)
            torch.cuda.synchronize()
            assert all(bool((t == 7.0).all()) for t in out), "outputs touched after a rejected layout"


def test_outputs_and_workspace_guard_bands(B):
    """Nothing is written outside dq/dk/dv or past the sized workspace."""
    wl = _wl("guard", torch.bfloat16, 1, 2, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=51)
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    o, lse = B.attn_forward(x["q"], x["k"], x["v"], scale=wl.scale, mask=wl.mask)
    g = 4096
    bufs = []
    for t in (x["q"], x["k"], x["v"]):
        big = torch.full((t.numel() + 2 * g,), float("nan"), dtype=t.dtype, device="cuda")
        bufs.append(big)
    outs = tuple(b[g:g + t.numel()].view(t.shape) for b, t in zip(bufs, (x["q"], x["k"], x["v"])))
    for det in (0, 1, 2):
        p = B.bwd_params(x["q"], x["k"], x["v"], o, x["do"], lse, *outs, scale=wl.scale, mask=wl.mask,
                         deterministic=det)
        need = B.workspace_bytes(p)
        ws = torch.full((need + 65536,), 0xAB, dtype=torch.uint8, device="cuda")
        assert B.attn_bwd(p, ws.data_ptr(), need, torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        assert (ws[need:] == 0xAB).all()
        for b, t in zip(bufs, outs):
            assert torch.isnan(b[:g]).all() and torch.isnan(b[-g:]).all()
            assert torch.isfinite(t).all()


def test_bounded_waits_expire_into_a_status(B):
    """Failure detection without a GPU fault: waits that can never end give up
    within their bound and report ATTN_ERR_TIMEOUT; a turn wait gives up at once
    when another CTA has already failed.  The context stays usable afterwards."""
    scratch = torch.zeros(B.SELFTEST_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    rc, status = B.attn_selftest_waits(scratch.data_ptr(), scratch.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert status == [-6, -6, 0], status
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0   # the device still works

