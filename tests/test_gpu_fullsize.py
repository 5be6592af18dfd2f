"""The benchmark workloads at full size, in the benchmark's launch
configuration (GPU forward, then attn_bwd through the C ABI), checked on
sampled rows that the fp64 oracle recomputes from Q, K, V and dO alone.
Packed THD workloads are checked segment by segment, every segment."""
import numpy as np
import pytest
import torch

from head_attention_backward_gb300 import workloads as W
from oracle import attn_ref as R
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


def _rows(n, rng, k=6):
    base = {0, 1, 63, 64, 127, 128, n // 2, n - 1}
    base |= set(int(v) for v in rng.integers(0, n, size=k))
    return sorted(r for r in base if 0 <= r < n)


def _run(B, wl, det):
    x = wl.inputs()
    cu = wl.cu_seqlens()
    d = {k: v.cuda() for k, v in x.items()}
    cu_d = None if cu is None else cu.cuda()
    cuk = wl.cu_seqlens_k()
    cuk_d = None if cuk is None else cuk.cuda()
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu_d,
              cu_seqlens_k=cuk_d, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o, lse = B.attn_forward(d["q"], d["k"], d["v"], **kw)
    got = B.attn_backward(d["q"], d["k"], d["v"], o, d["do"], lse, deterministic=det, **kw)
    torch.cuda.synchronize()
    return x, cu, [t.cpu() for t in got]


def _check_batch(wl, x, got, heads, kv_heads, seed):
    rng = np.random.default_rng(seed)
    okw = dict(mask=wl.mask, left=wl.left, right=wl.right)
    dq, dk, dv = got
    gq, rq, gk, rk, gv, rv = [], [], [], [], [], []
    for b, h in heads:
        rows = _rows(wl.sq, rng)
        rq.append(R.dq_rows(x["q"], x["k"], x["v"], x["do"], wl.scale, b, h, rows, **okw))
        gq.append(dq[b, rows, h])
    for b, hk in kv_heads:
        rows = _rows(wl.sk, rng)
        ek, ev = R.dkv_rows(x["q"], x["k"], x["v"], x["do"], wl.scale, b, hk, rows, **okw)
        rk.append(ek); rv.append(ev)
        gk.append(dk[b, rows, hk]); gv.append(dv[b, rows, hk])
    reps = []
    for name, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv)):
        rep = compare(torch.cat(g), torch.cat(r), 2e-2, 0.9999)
        rep["tensor"] = name
        reps.append(rep)
    return reps


def test_mha_causal_B4_H16_S2048(B):
    wl = W.mha_causal()
    for det in (False, True):
        x, _, got = _run(B, wl, det)
        assert_all_ok(_check_batch(wl, x, got, [(0, 0), (3, 15), (1, 7)], [(0, 0), (3, 15)], 1), f"det={det}")


@pytest.mark.parametrize("det", [1, 2], ids=["ordered", "split"])
def test_gqa_causal_det_B2_Hq32_Hkv8_S4096(B, det):
    wl = W.gqa_causal_det()
    x, _, got = _run(B, wl, det)
    assert_all_ok(_check_batch(wl, x, got, [(0, 0), (1, 31), (0, 13)], [(0, 0), (1, 7)], 2), f"gqa det={det}")


@pytest.mark.parametrize("det", [True, False], ids=["det", "atomic"])
def test_window_dqk192_dv128_S8192(B, det):
    wl = W.window_192(deterministic=det)
    x, _, got = _run(B, wl, det)
    assert_all_ok(_check_batch(wl, x, got, [(0, 0), (0, 15)], [(0, 5)], 5), f"window det={det}")


@pytest.mark.parametrize("det", [0, 1, 2], ids=["atomic", "ordered", "split"])
def test_head_dim_256_B1_Hq16_Hkv4_S4096(B, det):
    """Head dim 256: two passes per KV tile, one per column half of dK, dV, dQ,
    each pass a work item of its own (the ordered fold keeps turn counters
    per pass)."""
    wl = W.gqa_d256(deterministic=det)
    x, _, got = _run(B, wl, det)
    assert_all_ok(_check_batch(wl, x, got, [(0, 0), (0, 15), (0, 6)], [(0, 0), (0, 3)], 6), f"d256 det={det}")


@pytest.mark.parametrize("det", [1, 0], ids=["ordered", "atomic"])
def test_long_sequence_S131072_window_slices(B, det):
    """A 131,072-token sequence (its row, tile and LSE indices run far past the
    other workloads'; the split slices would need 137 GB here, so ordered fold
    and atomic only), window (1024, 0).  Each query row sees at most 1,025
    keys, so any 4,096-row slice starting on a tile boundary is self-contained
    for dQ rows 1,024 and up and for dK / dV key rows 1,024 to 3,071 (only
    queries inside the slice see them): those rows, in the first and in the
    last slice of the sequence, are compared with the oracle run on the slice
    alone."""
    wl = W.Workload("win_B1_Hq2_Hkv1_S131072_left1024", torch.bfloat16, 1, 2, 1, 131072, 131072, 128, 128,
                    W.MASK_WINDOW, left=1024, right=0, seed=61)
    x, _, got = _run(B, wl, det)
    dq, dk, dv = got
    okw = dict(mask=W.MASK_WINDOW, left=1024, right=0)
    rng = np.random.default_rng(61)
    for a in (0, 131072 - 4096):
        xs = {n: x[n][:, a:a + 4096] for n in ("q", "k", "v", "do")}
        qrows = sorted(set([1024, 1087, 2048, 4095]) | set(int(r) for r in rng.integers(1024, 4096, size=6)))
        krows = sorted(set([1024, 1151, 3071]) | set(int(r) for r in rng.integers(1024, 3072, size=5)))
        gq = torch.cat([dq[0, [a + r for r in qrows], h] for h in range(2)])
        rq = torch.cat([R.dq_rows(xs["q"], xs["k"], xs["v"], xs["do"], wl.scale, 0, h, qrows, **okw) for h in range(2)])
        ek, ev = R.dkv_rows(xs["q"], xs["k"], xs["v"], xs["do"], wl.scale, 0, 0, krows, **okw)
        reps = []
        for name, g, r in (("dq", gq, rq), ("dk", dk[0, [a + r for r in krows], 0], ek),
                           ("dv", dv[0, [a + r for r in krows], 0], ev)):
            rep = compare(g, r, 2e-2, 0.9999)
            rep["tensor"] = name
            reps.append(rep)
        assert_all_ok(reps, f"slice at {a}")


def test_head_dim_256_ordered_fold_equals_split_bits(B):
    wl = W.gqa_d256(deterministic=True)
    _, _, a = _run(B, wl, 1)
    _, _, b = _run(B, wl, 2)
    for name, x, y in zip(("dq", "dk", "dv"), a, b):
        assert torch.equal(x, y), name


@pytest.mark.parametrize("det", [0, 1, 2], ids=["atomic", "ordered", "split"])
def test_thd_packed_T16384_every_segment(B, det):
    """The packed THD workload's dq_acc slice (about 270 MB) is over the
    grouping threshold, so this also runs the grouped work order."""
    wl = W.thd_packed(deterministic=det)
    x, cu, (dq, dk, dv) = _run(B, wl, det)
    cu = cu.tolist()
    rng = np.random.default_rng(4)
    okw = dict(mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cu)
    reps = []
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b]
        rows = _rows(n, rng, k=4)
        idx = torch.tensor(rows) + cu[b]
        # two query heads (one random, one from the other half of the heads)
        # and both ends of the kv-head range, every segment
        h0 = int(rng.integers(0, wl.hq // 2))
        for h in (h0, h0 + wl.hq // 2):
            rq = R.dq_rows(x["q"], x["k"], x["v"], x["do"], wl.scale, b, h, rows, **okw)
            rep = compare(dq[idx, h], rq, 2e-2, 0.9999)
            rep.update(tensor="dq", segment=b, length=n, head=h)
            reps.append(rep)
        for hk in (0, wl.hkv - 1):
            ek, ev = R.dkv_rows(x["q"], x["k"], x["v"], x["do"], wl.scale, b, hk, rows, **okw)
            for name, g, r in (("dk", dk[idx, hk], ek), ("dv", dv[idx, hk], ev)):
                rep = compare(g, r, 2e-2, 0.9999)
                rep.update(tensor=name, segment=b, length=n, head=hk)
                reps.append(rep)
    assert_all_ok(reps, f"thd det={det}")


def test_thd_grouped_order_ordered_fold_equals_split_bits(B):
    """Under the grouped work order the ordered fold still adds each query
    tile's partials in ascending KV-tile order: same bits as the split slices."""
    wl = W.thd_packed(deterministic=True)
    _, _, a = _run(B, wl, 1)
    _, _, b = _run(B, wl, 2)
    for name, x, y in zip(("dq", "dk", "dv"), a, b):
        assert torch.equal(x, y), name


def test_bench_workload_deterministic_10_runs_bitwise(B):
    """The bench workload in both deterministic modes: 10 runs give the same
    bits, and the ordered fold gives the split slices' bits (compared on the
    device)."""
    wl = W.gqa_causal_det()
    x = {k: v.cuda() for k, v in wl.inputs().items()}
    kw = dict(scale=wl.scale, mask=wl.mask)
    o, lse = B.attn_forward(x["q"], x["k"], x["v"], **kw)
    first = {}
    for mode in (B.DET_ORDERED, B.DET_SPLIT):
        for i in range(10):
            got = B.attn_backward(x["q"], x["k"], x["v"], o, x["do"], lse, deterministic=mode, **kw)
            if i == 0:
                first[mode] = got
            else:
                for name, a, b in zip(("dq", "dk", "dv"), first[mode], got):
                    assert torch.equal(a, b), f"mode {mode} run {i}: {name} differs"
    for name, a, b in zip(("dq", "dk", "dv"), first[B.DET_ORDERED], first[B.DET_SPLIT]):
        assert torch.equal(a, b), f"ordered fold and split slices differ in {name}"


def test_forward_bitwise_repeatable_and_matches_oracle_full_size(B):
    """The tensor-core forward at the bench shape: eight calls give the same
    bits (all 2 x 4096 x 32 query rows; a race between the P/dS warps and the
    P V issuer shows as a few wrong 32-row groups in some calls only), and
    sampled heads match the fp64 forward."""
    wl = W.gqa_causal_det()
    x = wl.inputs()
    d = {k: v.cuda() for k, v in x.items()}
    kw = dict(scale=wl.scale, mask=wl.mask)
    o0, l0 = B.attn_forward(d["q"], d["k"], d["v"], **kw)
    for i in range(8):
        o, lse = B.attn_forward(d["q"], d["k"], d["v"], **kw)
        bad = int((o != o0).any(-1).sum())
        assert bad == 0 and torch.equal(lse, l0), f"call {i + 1}: {bad} O rows differ from the first call"
    o0, l0 = o0.cpu(), l0.cpu()
    vis = R.visible(wl.sq, wl.sk, wl.mask)
    reps = []
    for b, h in [(0, 0), (1, 17), (0, 30), (1, 5)]:
        hk = h // (wl.hq // wl.hkv)
        _, lse_ref, o_ref = R._head_forward(x["q"][b, :, h].double(), x["k"][b, :, hk].double(),
                                            x["v"][b, :, hk].double(), wl.scale, vis)
        rep = compare(o0[b, :, h], o_ref, 2e-2, 0.9999)
        rep.update(tensor="o", batch=b, head=h)
        reps.append(rep)
        rep = compare(l0[b, h], lse_ref, 2e-3, 0.9999)
        rep.update(tensor="lse", batch=b, head=h)
        reps.append(rep)
    assert_all_ok(reps, "forward full size")


@pytest.mark.parametrize("name", ["thd_packed", "window_192"])
def test_forward_bitwise_repeatable_other_workloads(B, name):
    """The forward on the packed THD and d_qk = 192 window workloads: five
    calls give the same bits."""
    wl = getattr(W, name)()
    d = {k: v.cuda() for k, v in wl.inputs().items()}
    cu = wl.cu_seqlens()
    cu = None if cu is None else cu.cuda()
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu, cu_seqlens_k=cu,
              max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o0, l0 = B.attn_forward(d["q"], d["k"], d["v"], **kw)
    for i in range(5):
        o, lse = B.attn_forward(d["q"], d["k"], d["v"], **kw)
        assert torch.equal(o, o0) and torch.equal(lse, l0), f"{name}: call {i + 1} differs from the first"


def test_window_dqk192_ordered_fold_equals_split_bits(B):
    wl = W.window_192(deterministic=True)
    _, _, a = _run(B, wl, 1)
    _, _, b = _run(B, wl, 2)
    for name, x, y in zip(("dq", "dk", "dv"), a, b):
        assert torch.equal(x, y), name


def test_bias_dropout_full_size_bitwise_repeatable(B):
    """The bias / dbias / dropout instantiation at a larger size (B1 Hq16 Hkv4
    S2048 d128 causal, a [1, Hq, S, S] bias, p = 0.1): five ordered-fold runs
    give the same bits, equal to the split slices' (values are checked against
    the oracle on small cases in test_gpu_extras.py)."""
    wl = W.Workload("bias_drop_B1_Hq16_S2048", torch.bfloat16, 1, 16, 4, 2048, 2048, 128, 128,
                    W.MASK_CAUSAL_TOP_LEFT, seed=31)
    d = {k: v.cuda() for k, v in wl.inputs().items()}
    g = torch.Generator().manual_seed(32)
    bias = torch.randn(1, wl.hq, wl.sq, wl.sk, generator=g).to(torch.bfloat16).cuda()
    seed = torch.tensor([1234], dtype=torch.int64, device="cuda")
    offset = torch.tensor([5], dtype=torch.int64, device="cuda")
    ex = dict(scale=wl.scale, mask=wl.mask, bias=bias, dropout_p=0.1, philox_seed=seed, philox_offset=offset)
    o, lse = B.attn_forward(d["q"], d["k"], d["v"], **ex)
    runs = {}
    for mode in (B.DET_ORDERED, B.DET_SPLIT):
        for i in range(5 if mode == B.DET_ORDERED else 1):
            got = B.attn_backward(d["q"], d["k"], d["v"], o, d["do"], lse, deterministic=mode, return_dbias=True, **ex)
            torch.cuda.synchronize()
            if mode not in runs:
                runs[mode] = got
            else:
                for name, a, b in zip(("dq", "dk", "dv", "dbias"), runs[mode], got):
                    assert torch.equal(a, b), f"run {i}: {name} differs"
    for name, a, b in zip(("dq", "dk", "dv", "dbias"), runs[B.DET_ORDERED], runs[B.DET_SPLIT]):
        assert torch.equal(a, b), f"ordered fold and split slices differ in {name}"
