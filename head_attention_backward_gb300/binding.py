"""ctypes binding of the C ABI in include/attn_bwd.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of ``libattn_bwd.so``;
this module only fills the parameter structs from torch tensors, allocates
outputs / workspace with torch (the library itself allocates nothing) and
passes the caller's current CUDA stream.  ``load()`` raises if the library has
not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_bwd.so")

ATTN_BF16, ATTN_FP16, ATTN_FP32 = 0, 1, 2
MASK_NONE, MASK_CAUSAL_TOP_LEFT, MASK_CAUSAL_BOTTOM_RIGHT, MASK_WINDOW = 0, 1, 2, 3
BIAS_NONE, BIAS_11SS, BIAS_1HSS, BIAS_BHSS, BIAS_B1SS = 0, 1, 2, 3, 4   # attn_bias_t
DET_ATOMIC, DET_ORDERED, DET_SPLIT = 0, 1, 2   # attn_det_t
STATUS = {0: "ATTN_OK", -1: "ATTN_ERR_INVALID_ARG", -2: "ATTN_ERR_UNSUPPORTED_HEADDIM",
          -3: "ATTN_ERR_WORKSPACE_TOO_SMALL", -4: "ATTN_ERR_CUDA", -5: "ATTN_ERR_DEVICE_FLAG",
          -6: "ATTN_ERR_TIMEOUT", -7: "ATTN_ERR_BAD_SEQLENS"}
# attn_status_t codes by name (ATTN_OK, ATTN_ERR_INVALID_ARG, ...)
globals().update({name: code for code, name in STATUS.items()})

_DTYPES = {torch.bfloat16: ATTN_BF16, torch.float16: ATTN_FP16, torch.float32: ATTN_FP32}

_i32, _vp, _f32 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
_i64x3 = ctypes.c_int64 * 3


class AttnBwdParams(ctypes.Structure):
    _fields_ = [("dtype", _i32), ("batch", _i32), ("nhead_q", _i32), ("nhead_kv", _i32),
                ("seqlen_q", _i32), ("seqlen_k", _i32), ("total_q", _i32), ("total_k", _i32),
                ("d_qk", _i32), ("d_v", _i32), ("cu_seqlens_q", _vp), ("cu_seqlens_k", _vp),
                ("cu_seqlens_q_padded", _vp), ("cu_seqlens_k_padded", _vp), ("mask", _i32), ("window_left", _i32), ("window_right", _i32),
                ("softmax_scale", _f32), ("deterministic", _i32),
                ("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("dout", _vp), ("lse", _vp),
                ("dq", _vp), ("dk", _vp), ("dv", _vp),
                ("stride_q", _i64x3), ("stride_k", _i64x3), ("stride_v", _i64x3), ("stride_o", _i64x3),
                ("stride_dout", _i64x3), ("stride_dq", _i64x3), ("stride_dk", _i64x3), ("stride_dv", _i64x3),
                ("bias_type", _i32), ("dropout_p", _f32), ("bias", _vp), ("dbias", _vp), ("philox_seed", _vp),
                ("philox_offset", _vp)]


class AttnFwdParams(ctypes.Structure):
    _fields_ = [("dtype", _i32), ("batch", _i32), ("nhead_q", _i32), ("nhead_kv", _i32),
                ("seqlen_q", _i32), ("seqlen_k", _i32), ("total_q", _i32), ("total_k", _i32),
                ("d_qk", _i32), ("d_v", _i32), ("cu_seqlens_q", _vp), ("cu_seqlens_k", _vp),
                ("cu_seqlens_q_padded", _vp), ("cu_seqlens_k_padded", _vp), ("mask", _i32), ("window_left", _i32), ("window_right", _i32),
                ("softmax_scale", _f32), ("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("lse", _vp),
                ("stride_q", _i64x3), ("stride_k", _i64x3), ("stride_v", _i64x3), ("stride_o", _i64x3),
                ("bias_type", _i32), ("dropout_p", _f32), ("bias", _vp), ("philox_seed", _vp), ("philox_offset", _vp)]


class AttnHostTensors(ctypes.Structure):
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("dout", _vp), ("lse", _vp),
                ("dq", _vp), ("dk", _vp), ("dv", _vp)]


EXPORTS = ["attn_bwd_workspace_size", "attn_bwd", "attn_bwd_timed", "attn_bwd_read_status",
           "attn_fwd", "attn_status_string", "attn_bwd_static_ws", "attn_selftest_waits", "attn_bwd_host"]

_lib = None


def load(path: str = LIB_PATH):
    """Load libattn_bwd.so and declare its signatures.  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -m head_attention_backward_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.attn_bwd_workspace_size.argtypes = [P(AttnBwdParams), P(ctypes.c_size_t)]
    lib.attn_bwd_workspace_size.restype = ctypes.c_int
    lib.attn_bwd.argtypes = [P(AttnBwdParams), _vp, ctypes.c_size_t, _vp]
    lib.attn_bwd.restype = ctypes.c_int
    lib.attn_bwd_timed.argtypes = [P(AttnBwdParams), _vp, ctypes.c_size_t, _vp, P(ctypes.c_float)]
    lib.attn_bwd_timed.restype = ctypes.c_int
    lib.attn_bwd_read_status.argtypes = [_vp, _vp, P(ctypes.c_int)]
    lib.attn_bwd_read_status.restype = ctypes.c_int
    lib.attn_fwd.argtypes = [P(AttnFwdParams), _vp]
    lib.attn_fwd.restype = ctypes.c_int
    lib.attn_status_string.argtypes = [ctypes.c_int]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_bwd_host.argtypes = [P(AttnBwdParams), P(AttnHostTensors), _vp, ctypes.c_size_t, _vp, _vp, _vp,
                                  ctypes.c_int]
    lib.attn_bwd_host.restype = ctypes.c_int
    _lib = lib
    return lib


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({attn_status_string(status)})")


# ------------------------------------------------------------ raw entry points

def attn_bwd_workspace_size(p: AttnBwdParams):
    n = ctypes.c_size_t(0)
    st = load().attn_bwd_workspace_size(ctypes.byref(p), ctypes.byref(n))
    return st, n.value


def attn_bwd(p: AttnBwdParams, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return load().attn_bwd(ctypes.byref(p), workspace, workspace_bytes, stream)


def attn_bwd_timed(p: AttnBwdParams, workspace: int, workspace_bytes: int, stream: int = 0):
    ms = (ctypes.c_float * 4)()
    st = load().attn_bwd_timed(ctypes.byref(p), workspace, workspace_bytes, stream, ms)
    return st, list(ms)


def attn_bwd_read_status(workspace: int, stream: int = 0):
    s = ctypes.c_int(0)
    st = load().attn_bwd_read_status(workspace, stream, ctypes.byref(s))
    return st, s.value


def attn_fwd(p: AttnFwdParams, stream: int = 0) -> int:
    return load().attn_fwd(ctypes.byref(p), stream)


def attn_bwd_host(p: AttnBwdParams, host: AttnHostTensors, workspace: int, workspace_bytes: int, stream: int,
                  copy_in: int, copy_out: int, chunks: int) -> int:
    return load().attn_bwd_host(ctypes.byref(p), ctypes.byref(host), workspace, workspace_bytes, stream, copy_in,
                                copy_out, chunks)


def host_tensors(q, k, v, o, do, lse, dq, dk, dv) -> AttnHostTensors:
    """Pinned host tensors (contiguous) for attn_bwd_host."""
    h = AttnHostTensors()
    for name, t in zip(("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv"), (q, k, v, o, do, lse, dq, dk, dv)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"host tensor {name} must be a contiguous CPU tensor (pinned for overlap)")
        setattr(h, name, t.data_ptr())
    return h


def attn_status_string(st: int) -> str:
    return load().attn_status_string(st).decode()


STATIC_WS_BYTES = 64 << 20


SELFTEST_SCRATCH_BYTES = 3 * 128 * 4 + 16


def attn_selftest_waits(scratch_ptr: int, scratch_bytes: int, stream: int = 0):
    """Runs the bounded-wait self-test; returns (rc, [status0, status1, status2])."""
    lib = load()
    fn = lib.attn_selftest_waits
    fn.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    fn.restype = ctypes.c_int
    out = (ctypes.c_int * 3)()
    rc = fn(ctypes.c_void_p(scratch_ptr), ctypes.c_size_t(scratch_bytes), ctypes.c_void_p(stream), out)
    return rc, list(out)


def attn_bwd_static_ws(p: AttnBwdParams, stream: int = 0) -> int:
    """attn_bwd with the library's own fixed device workspace: for callers
    that cannot allocate device memory.  Problems needing more than
    STATIC_WS_BYTES of workspace are rejected (ATTN_ERR_WORKSPACE_TOO_SMALL);
    calls overlapping on the GPU share that workspace and race."""
    lib = load()
    fn = lib.attn_bwd_static_ws
    fn.argtypes = [ctypes.POINTER(AttnBwdParams), _vp]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(p), stream)


# ------------------------------------------------------- tensor marshalling

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _strides(t, group: bool):
    """{batch, row, head} element strides of a [B,S,H,D] or [T,H,D] tensor
    whose last dimension is contiguous."""
    if t.stride(-1) != 1:
        raise ValueError("the head dimension must be contiguous (stride 1)")
    if group:
        return (0, t.stride(0), t.stride(1))
    return (t.stride(0), t.stride(1), t.stride(2))


def _set_strides(p, group: bool, **tensors):
    for name, t in tensors.items():
        getattr(p, "stride_" + name)[:] = _strides(t, group)


def _shape_args(q, k, v, cu_seqlens_q, max_seqlen_q, max_seqlen_k):
    if cu_seqlens_q is None:
        b, sq, hq, dqk = q.shape
        sk, hkv, dv = k.shape[1], k.shape[2], v.shape[3]
        return dict(batch=b, nhead_q=hq, nhead_kv=hkv, seqlen_q=sq, seqlen_k=sk, total_q=0,
                    total_k=0, d_qk=dqk, d_v=dv)
    tq, hq, dqk = q.shape
    tk, hkv, dv = k.shape[0], k.shape[1], v.shape[2]
    return dict(batch=cu_seqlens_q.numel() - 1, nhead_q=hq, nhead_kv=hkv, seqlen_q=max_seqlen_q,
                seqlen_k=max_seqlen_k, total_q=tq, total_k=tk, d_qk=dqk, d_v=dv)


def bias_type_of(bias: Optional[torch.Tensor], batch: int, nhead_q: int) -> int:
    """attn_bias_t of a [bias_b, bias_h, Sq, Sk] bias (bias_b in {1, B}, bias_h
    in {1, Hq})."""
    if bias is None:
        return BIAS_NONE
    bb, bh = bias.shape[0], bias.shape[1]
    if bias.dim() != 4 or bb not in (1, batch) or bh not in (1, nhead_q):
        raise ValueError("bias must be [1 or B, 1 or Hq, Sq, Sk]")
    if bb == 1 and bh == 1:
        return BIAS_11SS
    if bb == 1:
        return BIAS_1HSS
    return BIAS_B1SS if bh == 1 else BIAS_BHSS


def _set_extras(p, q, bias, dropout_p, philox_seed, philox_offset, dbias=None):
    if bias is not None:
        if not bias.is_contiguous():
            raise ValueError("the bias must be contiguous")
        p.bias_type = bias_type_of(bias, q.shape[0], q.shape[2])
        p.bias = bias.data_ptr()
    if dbias is not None:
        p.dbias = dbias.data_ptr()
    p.dropout_p = float(dropout_p)
    p.philox_seed, p.philox_offset = _ptr(philox_seed), _ptr(philox_offset)


def bwd_params(q, k, v, o, do, lse, dq, dk, dv, *, scale, mask=MASK_NONE, left=-1, right=-1,
               deterministic=False, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=0,
               max_seqlen_k=0, cu_seqlens_q_padded=None, cu_seqlens_k_padded=None, bias=None, dbias=None,
               dropout_p=0.0, philox_seed=None, philox_offset=None) -> AttnBwdParams:
    p = AttnBwdParams()
    p.dtype = _DTYPES[q.dtype]
    for name, val in _shape_args(q, k, v, cu_seqlens_q, max_seqlen_q, max_seqlen_k).items():
        setattr(p, name, val)
    p.cu_seqlens_q, p.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    p.cu_seqlens_q_padded, p.cu_seqlens_k_padded = _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_k_padded)
    p.mask, p.window_left, p.window_right = mask, left, right
    p.softmax_scale = scale
    p.deterministic = int(deterministic)   # False/True or an attn_det_t value (0, 1, 2)
    p.q, p.k, p.v, p.o, p.dout, p.lse = (_ptr(t) for t in (q, k, v, o, do, lse))
    p.dq, p.dk, p.dv = _ptr(dq), _ptr(dk), _ptr(dv)
    _set_strides(p, cu_seqlens_q is not None, q=q, k=k, v=v, o=o, dout=do, dq=dq, dk=dk, dv=dv)
    _set_extras(p, q, bias, dropout_p, philox_seed, philox_offset, dbias)
    return p


def fwd_params(q, k, v, o, lse, *, scale, mask=MASK_NONE, left=-1, right=-1, cu_seqlens_q=None,
               cu_seqlens_k=None, max_seqlen_q=0, max_seqlen_k=0, cu_seqlens_q_padded=None,
               cu_seqlens_k_padded=None, bias=None, dropout_p=0.0, philox_seed=None,
               philox_offset=None) -> AttnFwdParams:
    p = AttnFwdParams()
    p.dtype = _DTYPES[q.dtype]
    for name, val in _shape_args(q, k, v, cu_seqlens_q, max_seqlen_q, max_seqlen_k).items():
        setattr(p, name, val)
    p.cu_seqlens_q, p.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    p.cu_seqlens_q_padded, p.cu_seqlens_k_padded = _ptr(cu_seqlens_q_padded), _ptr(cu_seqlens_k_padded)
    p.mask, p.window_left, p.window_right = mask, left, right
    p.softmax_scale = scale
    p.q, p.k, p.v, p.o, p.lse = (_ptr(t) for t in (q, k, v, o, lse))
    _set_strides(p, cu_seqlens_q is not None, q=q, k=k, v=v, o=o)
    _set_extras(p, q, bias, dropout_p, philox_seed, philox_offset)
    return p


def workspace_bytes(p: AttnBwdParams) -> int:
    st, n = attn_bwd_workspace_size(p)
    if st != 0:
        raise AttnError(st, "attn_bwd_workspace_size")
    return n


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _empty_in_order_of(t, last: int):
    """An uninitialised tensor shaped like t but with last dimension `last`,
    its other dimensions laid out in t's memory order (so BHSD or SBHD inputs
    give a BHSD or SBHD output and the strides fold the same way)."""
    n = t.dim() - 1
    order = sorted(range(n), key=lambda i: -t.stride(i))
    buf = torch.empty([t.shape[i] for i in order] + [last], dtype=t.dtype, device=t.device)
    return buf.permute([order.index(i) for i in range(n)] + [n])


def attn_forward(q, k, v, *, scale, mask=MASK_NONE, left=-1, right=-1, cu_seqlens_q=None,
                 cu_seqlens_k=None, max_seqlen_q=0, max_seqlen_k=0, cu_seqlens_q_padded=None,
                 cu_seqlens_k_padded=None, stream=None, bias=None, dropout_p=0.0, philox_seed=None,
                 philox_offset=None):
    """O and LSE from the library's forward helper (outputs allocated here; the
    padding rows of a padded layout, which the helper leaves alone, hold O = 0
    and LSE = -inf)."""
    o = _empty_in_order_of(q, v.shape[-1])
    if cu_seqlens_q is None:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    else:
        o.zero_()
        lse = torch.full((q.shape[1], q.shape[0]), -math.inf, dtype=torch.float32, device=q.device)
    p = fwd_params(q, k, v, o, lse, scale=scale, mask=mask, left=left, right=right,
                   cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                   max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                   cu_seqlens_q_padded=cu_seqlens_q_padded, cu_seqlens_k_padded=cu_seqlens_k_padded,
                   bias=bias, dropout_p=dropout_p, philox_seed=philox_seed, philox_offset=philox_offset)
    st = attn_fwd(p, _stream(stream))
    if st != 0:
        raise AttnError(st, "attn_fwd")
    return o, lse


def attn_backward(q, k, v, o, do, lse, *, scale, mask=MASK_NONE, left=-1, right=-1,
                  deterministic=False, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=0,
                  max_seqlen_k=0, cu_seqlens_q_padded=None, cu_seqlens_k_padded=None,
                  workspace=None, out=None, stream=None, check_status=True, bias=None, return_dbias=False,
                  dropout_p=0.0, philox_seed=None, philox_offset=None):
    """dQ, dK, dV (and dbias [B, Hq, Sq, Sk] when return_dbias) through attn_bwd
    (outputs and workspace allocated here unless given).  `bias` is a
    [1 or B, 1 or Hq, Sq, Sk] tensor in the dtype of q; dropout takes a
    probability and one-element int64 device tensors for the philox seed and
    offset."""
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    dbias = None
    if return_dbias:
        dbias = torch.empty((q.shape[0], q.shape[2], q.shape[1], k.shape[1]), dtype=q.dtype, device=q.device)
    p = bwd_params(q, k, v, o, do, lse, dq, dk, dv, scale=scale, mask=mask, left=left, right=right,
                   deterministic=deterministic, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                   max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                   cu_seqlens_q_padded=cu_seqlens_q_padded, cu_seqlens_k_padded=cu_seqlens_k_padded,
                   bias=bias, dbias=dbias, dropout_p=dropout_p, philox_seed=philox_seed,
                   philox_offset=philox_offset)
    n = workspace_bytes(p)
    if workspace is None or workspace.numel() < n:
        workspace = alloc_workspace(n, q.device)
    s = _stream(stream)
    st = attn_bwd(p, workspace.data_ptr(), workspace.numel(), s)
    if st != 0:
        raise AttnError(st, "attn_bwd")
    if check_status:
        st, dev = attn_bwd_read_status(workspace.data_ptr(), s)
        if st != 0:
            raise AttnError(st, "attn_bwd_read_status")
        if dev != 0:
            raise AttnError(dev, "attn_bwd (device status)")
    if return_dbias:
        return dq, dk, dv, dbias
    return dq, dk, dv
