"""attn_bwd_static_ws: the entry point for callers that cannot allocate device
memory (its workspace is a fixed array inside the library).

It runs the same kernels in the same order as attn_bwd, so in the
deterministic modes its results must equal attn_bwd's bit for bit; in the
atomic mode (arrival-order fp32 sums) they are compared at the parity
tolerance.  The calls follow each other on the one shared array, mixing batch
and packed problems and all three dQ modes, so that state a call leaves behind
(turn counters, first-tile table, the zeroed slice, the status word) would
show up in the next one.  Collected last so that a failure here never hides
the rest of the suite."""
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
    """attn_bwd (caller workspace) and attn_bwd_static_ws on the same inputs."""
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
    assert st == B.ATTN_OK, B.attn_status_string(st)
    torch.cuda.synchronize()
    return outs, ref


def _check(B, wl, det, what):
    outs, ref = _case(B, wl, det)
    if det != B.DET_ATOMIC:
        for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
            assert torch.equal(g, r), f"{what}: {name} differs from attn_bwd"
        return
    reps = []
    for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
        rep = compare(g.cpu(), r.cpu(), 2e-2, 0.9999)
        rep["tensor"] = name
        reps.append(rep)
    assert_all_ok(reps, what)


def test_static_workspace_matches_attn_bwd_calls_in_a_row(B):
    batch = W.Workload("static_a", torch.bfloat16, 1, 4, 2, 300, 300, 128, 128, W.MASK_CAUSAL_TOP_LEFT,
                       seed=61)
    packed = W.thd("static_b", [100, 80, 76], hq=8, hkv=2, seed=62)
    _check(B, batch, B.DET_ORDERED, "first call (batch, ordered fold)")
    _check(B, packed, B.DET_ATOMIC, "second call (THD, atomic)")
    _check(B, batch, B.DET_SPLIT, "third call (batch, split slices)")
    _check(B, packed, B.DET_ORDERED, "fourth call (THD, ordered fold)")
    _check(B, batch, B.DET_ORDERED, "fifth call (batch, ordered fold again)")


def test_static_workspace_rejects_oversize_problem(B):
    """A problem whose workspace is larger than the array is refused before
    anything runs.  The tensors are real (uninitialised) device buffers of the
    problem's full size, so the test depends only on the size check."""
    b, hq, hkv, s, d = 1, 32, 8, 4096, 128
    q, o, do, dq = (torch.empty(b, s, hq, d, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    k, v, dk, dv = (torch.empty(b, s, hkv, d, dtype=torch.bfloat16, device="cuda") for _ in range(4))
    lse = torch.empty(b, hq, s, dtype=torch.float32, device="cuda")
    p = B.bwd_params(q, k, v, o, do, lse, dq, dk, dv, scale=d ** -0.5, mask=W.MASK_CAUSAL_TOP_LEFT,
                     deterministic=B.DET_ORDERED)
    assert B.workspace_bytes(p) > B.STATIC_WS_BYTES
    assert B.attn_bwd_static_ws(p, torch.cuda.current_stream().cuda_stream) == B.ATTN_ERR_WORKSPACE_TOO_SMALL
