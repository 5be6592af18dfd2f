"""C-ABI checks that need no GPU: the library loads, exports every function
include/attn_bwd.h declares, its ctypes mirrors match the C structs, the
workspace sizing is right, and every invalid configuration is rejected with
its error code before anything touches the device."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from head_attention_backward_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_bwd.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(attn_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(B.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def _c_layout():
    """sizeof / offsetof of the header's structs, from the C compiler."""
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "attn_bwd.h"
#define F(S, m) printf(#S "." #m " %zu\n", offsetof(S, m));
int main(void) {
  printf("attn_bwd_params.size %zu\n", sizeof(attn_bwd_params));
  printf("attn_fwd_params.size %zu\n", sizeof(attn_fwd_params));
  F(attn_bwd_params, cu_seqlens_q) F(attn_bwd_params, cu_seqlens_q_padded)
  F(attn_bwd_params, cu_seqlens_k_padded) F(attn_bwd_params, mask) F(attn_bwd_params, softmax_scale)
  F(attn_bwd_params, deterministic) F(attn_bwd_params, q) F(attn_bwd_params, lse) F(attn_bwd_params, dv)
  F(attn_bwd_params, stride_q) F(attn_bwd_params, stride_dout) F(attn_bwd_params, stride_dv)
  F(attn_fwd_params, stride_q) F(attn_fwd_params, stride_o)
  F(attn_bwd_params, bias_type) F(attn_bwd_params, dropout_p) F(attn_bwd_params, bias) F(attn_bwd_params, dbias)
  F(attn_bwd_params, philox_seed) F(attn_bwd_params, philox_offset)
  F(attn_fwd_params, bias_type) F(attn_fwd_params, dropout_p) F(attn_fwd_params, bias)
  F(attn_fwd_params, philox_seed) F(attn_fwd_params, philox_offset)
  printf("attn_host_tensors.size %zu\n", sizeof(attn_host_tensors));
  F(attn_host_tensors, lse) F(attn_host_tensors, dv)
  F(attn_fwd_params, cu_seqlens_k) F(attn_fwd_params, cu_seqlens_k_padded) F(attn_fwd_params, softmax_scale) F(attn_fwd_params, q) F(attn_fwd_params, lse)
  return 0;
}
"""
    tmp = os.path.join(ROOT, "head_attention_backward_gb300", "_build")
    os.makedirs(tmp, exist_ok=True)
    c = os.path.join(tmp, "layout.c")
    exe = os.path.join(tmp, "layout")
    open(c, "w").write(prog)
    cuda_inc = "/usr/local/cuda/include"
    r = subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, c, "-o", exe],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("gcc/CUDA headers unavailable: " + r.stderr[:200])
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}


def test_ctypes_structs_match_c_layout():
    lay = _c_layout()
    assert lay["attn_bwd_params.size"] == ctypes.sizeof(B.AttnBwdParams)
    assert lay["attn_fwd_params.size"] == ctypes.sizeof(B.AttnFwdParams)
    assert lay["attn_host_tensors.size"] == ctypes.sizeof(B.AttnHostTensors)
    classes = {"attn_bwd_params": B.AttnBwdParams, "attn_fwd_params": B.AttnFwdParams,
               "attn_host_tensors": B.AttnHostTensors}
    for key, off in lay.items():
        s, m = key.split(".")
        if m == "size":
            continue
        cls = classes[s]
        assert getattr(cls, m).offset == off, key


def make(**kw):
    p = B.AttnBwdParams()
    base = dict(dtype=B.ATTN_BF16, batch=2, nhead_q=32, nhead_kv=8, seqlen_q=4096, seqlen_k=4096,
                total_q=0, total_k=0, d_qk=128, d_v=128, mask=1, window_left=-1, window_right=-1,
                softmax_scale=0.088, deterministic=1)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    # fake, 16-byte aligned addresses: validation never dereferences them
    for i, name in enumerate(["q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"]):
        if getattr(p, name) is None and name not in kw:
            setattr(p, name, 0x10000 * (i + 1))
    return p


def test_workspace_size_split_holds_all_splits(lib):
    st, n = B.attn_bwd_workspace_size(make(deterministic=B.DET_SPLIT))
    assert st == 0
    nsplits = 4096 // 128
    dq_acc = nsplits * 2 * 32 * 4096 * 128 * 4
    assert dq_acc <= n < dq_acc + 16 * 2**20


def test_workspace_size_ordered_fold_one_slice_plus_turns(lib):
    st, n = B.attn_bwd_workspace_size(make(deterministic=B.DET_ORDERED))
    assert st == 0
    one = 2 * 32 * 4096 * 128 * 4
    turns = 32 * 2 * (4096 // 64) * 4
    assert one + turns <= n < one + 16 * 2**20


def test_workspace_size_fp32_ordered_uses_split_slices(lib):
    st, n = B.attn_bwd_workspace_size(make(dtype=B.ATTN_FP32, d_qk=64, d_v=64, deterministic=B.DET_ORDERED))
    assert st == 0
    assert n >= (4096 // 128) * 2 * 32 * 4096 * 64 * 4


def test_workspace_size_head_dim_256_ordered_folds_into_one_slice(lib):
    """d_qk = 256 runs two passes per KV tile (one per column half); the
    ordered fold keeps one slice, with a turn counter per pass, head and
    query tile."""
    st, n = B.attn_bwd_workspace_size(make(d_qk=256, d_v=256, deterministic=B.DET_ORDERED))
    assert st == 0
    one = 2 * 32 * 4096 * 256 * 4
    assert one <= n < one + 16 * 2**20
    st, n_split = B.attn_bwd_workspace_size(make(d_qk=256, d_v=256, deterministic=B.DET_SPLIT))
    assert st == 0 and n_split >= (4096 // 128) * one


def test_workspace_size_atomic_one_slice(lib):
    st, n = B.attn_bwd_workspace_size(make(deterministic=0))
    assert st == 0
    one = 2 * 32 * 4096 * 128 * 4
    assert one <= n < one + 16 * 2**20


def test_workspace_size_group_mode(lib):
    p = make(deterministic=B.DET_SPLIT, batch=3, seqlen_q=300, seqlen_k=300, total_q=700, total_k=700)
    p.cu_seqlens_q = 0x1000
    p.cu_seqlens_k = 0x2000
    st, n = B.attn_bwd_workspace_size(p)
    assert st == 0
    nsplits = (300 + 127) // 128
    assert n >= nsplits * 32 * 700 * 128 * 4


def test_workspace_size_is_pure_host_arithmetic(lib):
    # same answer twice and for null tensor pointers: no device access involved
    p = make()
    for name in ["q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"]:
        setattr(p, name, None)
    a = B.attn_bwd_workspace_size(p)
    b = B.attn_bwd_workspace_size(make())
    assert a == b and a[0] == 0


ERR = dict(inv=-1, hd=-2, ws=-3)


@pytest.mark.parametrize("kw,code", [
    (dict(nhead_q=30, nhead_kv=8), "inv"),
    (dict(batch=0), "inv"),
    (dict(dtype=7), "inv"),
    (dict(mask=9), "inv"),
    (dict(deterministic=3), "inv"),
    (dict(deterministic=-1), "inv"),
    (dict(mask=3, window_left=-2), "inv"),
    (dict(softmax_scale=float("nan")), "inv"),
    (dict(seqlen_q=-1), "inv"),
    (dict(d_qk=96, d_v=96), "hd"),
    (dict(d_qk=128, d_v=64), "hd"),
    (dict(dtype=B.ATTN_FP32, d_qk=128, d_v=128), "hd"),
    (dict(d_qk=256, d_v=128), "hd"),
    (dict(d_qk=320, d_v=320), "hd"),
    (dict(dtype=B.ATTN_FP32, d_qk=256, d_v=256), "hd"),
    (dict(q=None), "inv"),
    (dict(dq=0x10008), "inv"),          # not 16-byte aligned
    (dict(bias_type=5, bias=0x200000), "inv"),               # unknown bias shape
    (dict(bias_type=1), "inv"),                              # bias shape without a bias
    (dict(bias_type=1, bias=0x200001), "inv"),               # bias not 2-byte aligned
    (dict(dbias=0x300000), "inv"),                           # dbias without a bias
    (dict(dtype=B.ATTN_FP32, d_qk=64, d_v=64, bias_type=3, bias=0x200000), "inv"),   # extras: 16-bit only
    (dict(dropout_p=1.0, philox_seed=0x400000, philox_offset=0x400008), "inv"),
    (dict(dropout_p=-0.1, philox_seed=0x400000, philox_offset=0x400008), "inv"),
    (dict(dropout_p=float("nan"), philox_seed=0x400000, philox_offset=0x400008), "inv"),
    (dict(dropout_p=0.5), "inv"),                            # no philox seed / offset
    (dict(dropout_p=0.5, philox_seed=0x400004, philox_offset=0x400008), "inv"),   # seed not 8-byte aligned
])
def test_invalid_arguments_rejected_before_launch(lib, kw, code):
    p = make(**kw)
    st = B.attn_bwd(p, 0x100000, 1 << 40, 0)
    assert st == ERR[code], (kw, st)


def test_bias_rejected_in_group_mode(lib):
    """The attention bias is defined for batch mode only (TE PR #446 sets the
    bias shape only outside group mode)."""
    p = make(total_q=100, total_k=100, bias_type=1, bias=0x200000)
    p.cu_seqlens_q, p.cu_seqlens_k = 0x1000, 0x2000
    assert B.attn_bwd(p, 0x100000, 1 << 40, 0) == -1


def test_group_mode_needs_both_seqstart_arrays(lib):
    p = make(total_q=100, total_k=100)
    p.cu_seqlens_q = 0x1000           # cu_seqlens_k left NULL
    assert B.attn_bwd_workspace_size(p)[0] == -1
    assert B.attn_bwd(p, 0x100000, 1 << 40, 0) == -1


def test_seqstart_arrays_must_be_int32_aligned(lib):
    p = make(total_q=100, total_k=100)
    p.cu_seqlens_q, p.cu_seqlens_k = 0x1000, 0x2000
    assert B.attn_bwd_workspace_size(p)[0] == 0
    for field in ("cu_seqlens_q", "cu_seqlens_k", "cu_seqlens_q_padded", "cu_seqlens_k_padded"):
        q = make(total_q=100, total_k=100)
        q.cu_seqlens_q, q.cu_seqlens_k = 0x1000, 0x2000
        setattr(q, field, 0x3002)
        assert B.attn_bwd_workspace_size(q)[0] == -1, field
        assert B.attn_bwd(q, 0x100000, 1 << 40, 0) == -1, field


def _with_strides(p, **strides):
    for name, val in strides.items():
        getattr(p, "stride_" + name)[:] = val
    return p


def test_strides_validated(lib):
    S, H, Hk, D = 4096, 32, 8, 128
    # BHSD ([B,H,S,D] buffers seen as [B,S,H,D]) on every tensor: batch folded into heads
    bh = dict(q=(H * S * D, D, S * D), k=(Hk * S * D, D, S * D), v=(Hk * S * D, D, S * D),
              o=(H * S * D, D, S * D), dout=(H * S * D, D, S * D), dq=(H * S * D, D, S * D),
              dk=(Hk * S * D, D, S * D), dv=(Hk * S * D, D, S * D))
    ok, n_bhsd = B.attn_bwd_workspace_size(_with_strides(make(), **bh))
    assert ok == 0 and 0 < n_bhsd <= B.attn_bwd_workspace_size(make())[1]
    # BHSD on q alone, the rest BSHD: the batch cannot be folded one way for all
    assert B.attn_bwd_workspace_size(_with_strides(make(), q=bh["q"]))[0] == -1
    # packed QKV rows (batch stride = S x row stride) mix with contiguous tensors
    assert B.attn_bwd_workspace_size(_with_strides(make(), q=(S * 3 * H * D, 3 * H * D, D)))[0] == 0
    bad = [(0, H * D, D),                             # batch stride missing with B = 2
           (S * H * D, H * D + 4, D),                 # 16-bit row stride not a multiple of 8
           (S * H * D, H * D, -D),                    # negative head stride
           (S * H * D, 1 << 37, D)]                   # beyond the tensor-map stride range
    for st in bad:
        assert B.attn_bwd_workspace_size(_with_strides(make(), q=st))[0] == -1, st
        assert B.attn_bwd(_with_strides(make(), dq=st), 0x100000, 1 << 40, 0) == -1, st
        assert B.attn_bwd(_with_strides(make(), dv=st), 0x100000, 1 << 40, 0) == -1, st
    # fp32 tensors take any positive stride; group mode ignores the batch stride
    p = _with_strides(make(dtype=B.ATTN_FP32, d_qk=32, d_v=33), q=(S * (H * 32 + 1), H * 32 + 1, 32))
    assert B.attn_bwd_workspace_size(p)[0] == 0
    p = _with_strides(make(total_q=100, total_k=100), q=(0, H * D, D))
    p.cu_seqlens_q, p.cu_seqlens_k = 0x1000, 0x2000
    assert B.attn_bwd_workspace_size(p)[0] == 0


def test_strided_test_layouts_are_accepted(lib):
    """Every strided layout the GPU parity tests use passes the sizing call's
    stride checks (batch folded along rows or heads), and a tensor set that
    mixes the two foldings is refused."""
    from head_attention_backward_gb300 import workloads as W
    from tests.parity import STRIDED_LAYOUTS, layout_heads_outer
    cases = [W.Workload("b", torch.bfloat16, 2, 4, 2, 300, 300, 128, 128, 1),
             W.Workload("b1", torch.bfloat16, 3, 4, 1, 200, 333, 64, 64, 0),
             W.Workload("f", torch.float32, 2, 2, 1, 150, 150, 64, 64, 1),
             W.thd("t", [100, 0, 37], hq=4, hkv=2, gaps_q=[1, 0, 2, 3], gaps_k=[0, 0, 0, 5])]
    for wl in cases:
        x = wl.inputs()
        x["o"] = torch.zeros_like(x["do"])
        cu = wl.cu_seqlens()
        kw = {}
        if cu is not None:
            kw = dict(cu_seqlens_q=cu, cu_seqlens_k=wl.cu_seqlens_k(), cu_seqlens_q_padded=wl.cu_seqlens_q_padded(),
                      cu_seqlens_k_padded=wl.cu_seqlens_k_padded())
        lse = torch.zeros(wl.shapes()["lse"])
        for layout in STRIDED_LAYOUTS:
            if layout.__name__ == "layout_sbhd" and wl.group_mode:
                continue
            if layout.__name__ == "layout_packed" and (x["q"].shape[:-2] != x["k"].shape[:-2] or wl.d_qk != wl.d_v):
                continue   # one packed buffer holds q, k and v rows side by side
            ins, out = layout(x)
            p = B.bwd_params(ins["q"], ins["k"], ins["v"], ins["o"], ins["do"], lse, *out, scale=0.1, mask=wl.mask,
                             max_seqlen_q=wl.sq, max_seqlen_k=wl.sk, **kw)
            assert B.attn_bwd_workspace_size(p)[0] == 0, (wl.name, layout.__name__)
        if not wl.group_mode and wl.batch > 1:
            ins, out = layout_heads_outer(x)
            p = B.bwd_params(ins["q"], ins["k"], ins["v"], x["o"], x["do"], lse, *out, scale=0.1, mask=wl.mask)
            assert B.attn_bwd_workspace_size(p)[0] == -1, wl.name


def test_host_entry_validates_before_launch(lib):
    def host(**kw):
        h = B.AttnHostTensors()
        for i, name in enumerate(["q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"]):
            setattr(h, name, kw.get(name, 0x20000 * (i + 1)))
        return h
    ws, n = 0x100000, 1 << 40
    assert B.attn_bwd_host(make(), host(lse=0), ws, n, 1, 2, 3, 2) == -1          # missing host tensor
    assert B.attn_bwd_host(make(), host(), ws, n, 1, 1, 3, 2) == -1               # streams not distinct
    assert B.attn_bwd_host(make(), host(), ws, n, 1, 2, 2, 2) == -1
    assert B.attn_bwd_host(_with_strides(make(), q=(4096 * 3 * 32 * 128, 3 * 32 * 128, 128)), host(),
                           ws, n, 1, 2, 3, 2) == -1                                # staging must be contiguous
    assert B.attn_bwd_host(make(), host(), ws, 1024, 1, 2, 3, 2) == -3            # workspace too small
    assert B.attn_bwd_host(make(d_qk=96, d_v=96), host(), ws, n, 1, 2, 3, 2) == -2


def test_padded_starts_only_in_group_mode(lib):
    p = make()                        # batch mode
    p.cu_seqlens_q_padded = 0x1000
    assert B.attn_bwd_workspace_size(p)[0] == -1
    assert B.attn_bwd(p, 0x100000, 1 << 40, 0) == -1
    p = make()
    p.cu_seqlens_k_padded = 0x1000
    assert B.attn_bwd(p, 0x100000, 1 << 40, 0) == -1


def test_workspace_too_small_and_misaligned(lib):
    p = make()
    _, need = B.attn_bwd_workspace_size(p)
    assert B.attn_bwd(p, 0x100000, need - 1, 0) == -3
    assert B.attn_bwd(p, 0x100010, need, 0) == -1      # not 256-byte aligned
    assert B.attn_bwd(p, None, need, 0) == -1


def test_null_params_and_status_strings(lib):
    assert lib.attn_bwd(None, None, 0, None) == -1
    n = ctypes.c_size_t(1)
    assert lib.attn_bwd_workspace_size(None, ctypes.byref(n)) == -1 and n.value == 0
    for code in [0, -1, -2, -3, -4, -5, -6, -7]:
        s = B.attn_status_string(code)
        assert s and s != "unknown status"
    assert B.attn_status_string(-99) == "unknown status"


def test_fwd_rejects_bad_args(lib):
    p = B.AttnFwdParams()
    p.dtype, p.batch, p.nhead_q, p.nhead_kv, p.seqlen_q, p.seqlen_k = 0, 1, 4, 3, 16, 16
    p.d_qk, p.d_v, p.softmax_scale = 64, 64, 0.1
    assert B.attn_fwd(p, 0) == -1          # 4 % 3 != 0
    p.nhead_kv = 2
    assert B.attn_fwd(p, 0) == -1          # null pointers
    p.q, p.k, p.v, p.o, p.lse = 0x1000, 0x2000, 0x3000, 0x4000, 0x5000
    p.d_qk = 320
    assert B.attn_fwd(p, 0) == -2
    p.d_qk = 64
    p.o = 0x4002                           # O is written with 16-byte vector stores
    assert B.attn_fwd(p, 0) == -1
    p.o, p.q = 0x4000, 0x1008              # q feeds a tensor map
    assert B.attn_fwd(p, 0) == -1
    p.q, p.lse = 0x1000, 0x5002            # lse: 4-byte alignment
    assert B.attn_fwd(p, 0) == -1
    p.dtype, p.lse, p.o = 2, 0x5000, 0x4004   # fp32: 4-byte alignment is enough, 2 is not
    p.q = 0x1002
    assert B.attn_fwd(p, 0) == -1
