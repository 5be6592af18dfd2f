"""Small ragged, windowed and GQA cases run on the -DATTN_DEBUG build of the
library (device-side index checks at every computed address).  Run as a
child process by tests/test_gpu_debug_build.py, so that the debug library is
the only one loaded in it.  Exits non-zero on the first failed case."""
import sys

import torch

sys.path.insert(0, __file__.rsplit("/tests/", 1)[0])
from head_attention_backward_gb300 import binding as B  # noqa: E402
from head_attention_backward_gb300 import build, workloads as W  # noqa: E402
from oracle import attn_ref as R  # noqa: E402
from tests.parity import assert_all_ok, call_scale, compare, per_segment_report, tolerances  # noqa: E402


def case_list():
    wl = lambda *a, **k: W.Workload(*a, **k)
    return [
        W.thd("thd_ragged", [1, 1, 130, 1, 100, 80, 76], hq=4, hkv=2, seed=91),
        wl("win192", torch.bfloat16, 1, 2, 2, 300, 300, 192, 128, W.MASK_WINDOW, 70, 0, False, 92, None),
        wl("br_short_k", torch.bfloat16, 1, 2, 1, 200, 90, 128, 128, W.MASK_CAUSAL_BOTTOM_RIGHT, -1, -1, False, 93, None),
        wl("nomask_sq_ne_sk", torch.bfloat16, 2, 2, 2, 70, 150, 64, 64, W.MASK_NONE, -1, -1, False, 94, None),
        wl("fp32", torch.float32, 1, 2, 1, 150, 150, 64, 64, W.MASK_CAUSAL_TOP_LEFT, -1, -1, False, 95, None),
        W.thd("thd_cross_br", [100, 0, 37, 250, 5], hq=4, hkv=2, mask=W.MASK_CAUSAL_BOTTOM_RIGHT,
              seed=96, seqlens_k=[300, 64, 0, 129, 200]),
        W.thd("thd_padded", [100, 0, 37, 250, 5], hq=4, hkv=2, mask=W.MASK_CAUSAL_BOTTOM_RIGHT,
              seed=97, seqlens_k=[300, 64, 0, 129, 200], gaps_q=[3, 0, 17, 140, 2, 9],
              gaps_k=[0, 5, 131, 7, 1, 30]),
        wl("d256", torch.bfloat16, 1, 2, 1, 200, 200, 256, 256, W.MASK_CAUSAL_TOP_LEFT, -1, -1, False, 98, None),
        wl("bias_dropout", torch.bfloat16, 2, 4, 2, 150, 150, 128, 128, W.MASK_CAUSAL_TOP_LEFT, -1, -1, False, 99,
           None),
    ]


# extras per case: a [B, Hq, Sq, Sk] bias with dbias, and dropout
EXTRAS = {"bias_dropout": dict(dropout_p=0.25, seed=5, offset=9)}


def main():
    B.load(build.build_library(variant="debug"))
    for w in case_list():
        x = w.inputs()
        cu, cuk = w.cu_seqlens(), w.cu_seqlens_k()
        stq, stk = w.cu_seqlens_q_padded(), w.cu_seqlens_k_padded()
        kw = dict(mask=w.mask, left=w.left, right=w.right, cu_seqlens_q=cu, cu_seqlens_k=cuk)
        if stq is not None or stk is not None:
            kw.update(cu_seqlens_q_padded=stq, cu_seqlens_k_padded=stk)
        ex = EXTRAS.get(w.name)
        okw, gkw = dict(kw), {}
        if ex:
            g = torch.Generator().manual_seed(w.seed)
            bias = torch.randn((w.batch, w.hq, w.sq, w.sk), generator=g).to(w.dtype)
            okw.update(bias=bias, dropout_p=ex["dropout_p"], philox_seed=ex["seed"], philox_offset=ex["offset"])
            gkw = dict(bias=bias.cuda(), return_dbias=True, dropout_p=ex["dropout_p"],
                       philox_seed=torch.tensor([ex["seed"]], dtype=torch.int64, device="cuda"),
                       philox_offset=torch.tensor([ex["offset"]], dtype=torch.int64, device="cuda"))
        o64, lse64 = R.attn_forward(x["q"], x["k"], x["v"], w.scale, **okw)
        o_in, lse_in = o64.to(w.dtype), lse64.to(torch.float32)
        ref = R.attn_backward(x["q"], x["k"], x["v"], o_in, x["do"], lse_in, w.scale, return_dbias=bool(ex), **okw)
        d = {k: v.cuda() for k, v in x.items()}
        dkw = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
        tol, mcos = tolerances(w.dtype)
        for mode in (0, 1, 2):
            got = B.attn_backward(d["q"], d["k"], d["v"], o_in.cuda(), d["do"], lse_in.cuda(), scale=w.scale,
                                  deterministic=mode, max_seqlen_q=w.sq, max_seqlen_k=w.sk, **dkw, **gkw)
            torch.cuda.synchronize()
            reps = []
            cf = call_scale(ref)
            for name, g, r in zip(("dq", "dk", "dv", "dbias"), got, ref):
                rep = compare(g.cpu(), r, tol, mcos, cf)
                rep["tensor"] = name
                reps.append(rep)
                if cu is not None:
                    offs, st = (cu, stq) if name == "dq" else (cuk, stk)
                    reps.extend(per_segment_report(g.cpu(), r, offs.tolist(), name, tol, mcos,
                                                   None if st is None else st.tolist(), call_floor=cf))
            assert_all_ok(reps, f"{w.name} mode {mode} (debug build)")
            print(f"ok {w.name} mode {mode}")


if __name__ == "__main__":
    main()
