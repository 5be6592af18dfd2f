"""attn_bwd_static_ws: the entry point for callers that cannot allocate device
memory (its workspace is a fixed array inside the library).  Checked against
the allocating entry point attn_bwd on the same inputs, on two calls in a row
that reuse the shared array, within the parity tolerance of the other tests.
Collected last so that a failure here never hides the rest of the suite."""
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from tests.parity import assert_all_ok, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_attention_backward_gb300 import build, binding
    build.build_library()
    binding.load()
    return binding


def _case(B, wl, det):
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    cu = wl.cu_seqlens()
    cu_d = None if cu is None else cu.cuda()
    cuk = wl.cu_seqlens_k()
    cuk_d = None if cuk is None else cuk.cuda()
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu_d,
              cu_seqlens_k=cuk_d, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o, lse = B.attn_forward(x["q"], x["k"], x["v"], **kw)
    ref = B.attn_backward(x["q"], x["k"], x["v"], o, x["do"], lse, deterministic=det, **kw)
    outs = (torch.full_like(x["q"], float("nan")), torch.full_like(x["k"], float("nan")),
            torch.full_like(x["v"], float("nan")))
    p = B.bwd_params(x["q"], x["k"], x["v"], o, x["do"], lse, *outs, deterministic=det, **kw)
    assert B.workspace_bytes(p) <= B.STATIC_WS_BYTES
    st = B.attn_bwd_static_ws(p, torch.cuda.current_stream().cuda_stream)
    assert st == 0, B.attn_status_string(st)
    torch.cuda.synchronize()
    reps = []
    for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
        rep = compare(g.cpu(), r.cpu(), 2e-2, 0.9999)
        rep["tensor"] = name
        reps.append(rep)
    return reps


def test_static_workspace_matches_attn_bwd_two_calls_in_a_row(B):
    batch = W.Workload("static_a", torch.bfloat16, 1, 4, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT,
                       seed=61)
    packed = W.thd("static_b", [100, 80, 76], hq=8, hkv=2, seed=62)
    assert_all_ok(_case(B, batch, True), "first call (batch, deterministic)")
    assert_all_ok(_case(B, packed, False), "second call (THD, atomic)")
    assert_all_ok(_case(B, batch, True), "third call (batch again)")


def test_static_workspace_rejects_oversize_problem(B):
    p = B.AttnBwdParams()
    for k, v in dict(dtype=0, batch=2, nhead_q=32, nhead_kv=8, seqlen_q=4096, seqlen_k=4096, d_qk=128,
                     d_v=128, mask=1, softmax_scale=0.088, deterministic=1).items():
        setattr(p, k, v)
    for i, name in enumerate(["q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"]):
        setattr(p, name, 0x10000 * (i + 1))
    assert B.attn_bwd_static_ws(p, 0) == -3
