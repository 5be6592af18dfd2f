"""attn_bwd_host: host tensors in, gradients back in host memory, the batch
split into chunks whose copies overlap the neighbouring chunks' compute.
The deterministic modes must give the same bits as one attn_bwd call on the
device; the atomic mode must match the oracle."""
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from oracle import attn_ref as R
from tests.parity import assert_all_ok, compare, tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_backward_gb300 import build, binding
    build.build_library()
    binding.load()
    return binding


def _case(wl):
    x = wl.inputs()
    cu, cuk = wl.cu_seqlens(), wl.cu_seqlens_k()
    kw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    if wl.gaps_q or wl.gaps_k:
        kw.update(cu_seqlens_q_padded=wl.cu_seqlens_q_padded(), cu_seqlens_k_padded=wl.cu_seqlens_k_padded())
    o, lse = R.attn_forward(x["q"], x["k"], x["v"], wl.scale, **kw)
    x["o"], x["lse"] = o.to(wl.dtype), lse.to(torch.float32)
    return x, kw


def _host_run(B, wl, x, kw, det, chunks):
    dev = {n: torch.empty_like(t, device="cuda") for n, t in x.items()}   # staging, filled by the call
    outs = tuple(torch.full_like(dev[n], float("nan")) for n in ("q", "k", "v"))
    dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    p = B.bwd_params(dev["q"], dev["k"], dev["v"], dev["o"], dev["do"], dev["lse"], *outs, scale=wl.scale,
                     deterministic=det, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, **dkw)
    ws = torch.empty(max(B.workspace_bytes(p), 256), dtype=torch.uint8, device="cuda")
    host_in = {n: t.contiguous().pin_memory() for n, t in x.items()}
    host_out = tuple(torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for t in outs)
    h = B.host_tensors(host_in["q"], host_in["k"], host_in["v"], host_in["o"], host_in["do"], host_in["lse"],
                       *host_out)
    s, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    rc = B.attn_bwd_host(p, h, ws.data_ptr(), ws.numel(), s.cuda_stream, s_in.cuda_stream, s_out.cuda_stream,
                         chunks)
    assert rc == 0, B.attn_status_string(rc)
    s.synchronize()
    st, status = B.attn_bwd_read_status(ws.data_ptr(), s.cuda_stream)
    assert st == 0 and status == 0, status
    return host_out


def _device_run(B, wl, x, kw, det):
    dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    d = {n: t.cuda() for n, t in x.items()}
    got = B.attn_backward(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], scale=wl.scale, deterministic=det,
                          max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, **dkw)
    torch.cuda.synchronize()
    return tuple(t.cpu() for t in got)


CASES = [
    W.Workload("gqa_b3_causal", torch.bfloat16, 3, 4, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT, seed=71),
    W.Workload("mha_b4_window_d64", torch.bfloat16, 4, 2, 2, 257, 257, 64, 64, W.MASK_WINDOW, 40, 0, seed=72),
    W.thd("thd", [100, 0, 37, 250, 5], hq=4, hkv=2, seed=73),
    W.thd("thd_cross_padded", [100, 0, 37], hq=6, hkv=3, mask=W.MASK_CAUSAL_BOTTOM_RIGHT, seed=74,
          seqlens_k=[300, 64, 0], gaps_q=[3, 0, 17, 5], gaps_k=[0, 5, 131, 2]),
]


@pytest.mark.parametrize("det", [1, 2], ids=["ordered", "split"])
@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_host_entry_bitwise_equal_to_device_call(B, wl, det):
    x, kw = _case(wl)
    ref = _device_run(B, wl, x, kw, det)
    # chunks beyond the batch split the kv heads too (2-D copies of head slices)
    for chunks in (1, 2, 3, 8):
        got = _host_run(B, wl, x, kw, det, chunks)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), f"{wl.name} chunks={chunks} {name}"


def test_host_entry_atomic_matches_oracle(B):
    wl = CASES[0]
    x, kw = _case(wl)
    ref = R.attn_backward(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], wl.scale, **kw)
    got = _host_run(B, wl, x, kw, 0, 3)
    tol, mcos = tolerances(wl.dtype)
    reps = [dict(compare(g, r, tol, mcos), tensor=n) for n, g, r in zip(("dq", "dk", "dv"), got, ref)]
    assert_all_ok(reps, "attn_bwd_host atomic")
