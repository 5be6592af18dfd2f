"""Benchmark of the FMHA backward on the Llama-3-8B-shaped GQA workload.

Default workload: B=2, Hq=32, Hkv=8, S=4096, d=128, causal, deterministic
dQ (the per-KV-tile partials summed in ascending KV-tile order: the ordered
fold by default; the split workspace of nsplits = 32 dq_acc slices plus a
reduction kernel is timed beside it and gives the same bits), bf16 inputs
~ N(0, 1), O/LSE from the forward helper.  One step = one whole attn_bwd call (schedule, preprocess, main
kernel, dQ reduce/convert) on inputs resident in HBM; L2 is flushed (256 MB
write) before every timed step.  Metric: mask-adjusted TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica on its own GPU (the
method has no cross-GPU exchange); the value is the whole-job throughput,
timed as the max over ranks.  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from head_attention_backward_gb300 import flops as FL  # noqa: E402
from head_attention_backward_gb300 import workloads as W  # noqa: E402

METRIC = "attn-bwd TFLOP/s (mask-adjusted, bf16) and % of GB300 dense BF16 peak"
WORKLOADS = {"gqa_causal_det": W.gqa_causal_det, "mha_causal": W.mha_causal,
             "thd_packed": W.thd_packed, "window_192": W.window_192, "gqa_d256": W.gqa_d256}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, pg=None, device="cpu"):
    """Element-wise max of a list of floats over all ranks (timings only;
    the method itself exchanges no data between GPUs)."""
    if pg is None:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world, flops_per_replica, ms_per_step):
    """Whole-job TFLOP/s: every rank runs one replica per step; the step time
    is the slowest rank's."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1900.0), d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 6800.0, "fallback"


# DRAM bytes (read + write) per launch of the main kernel, from a one-pass ncu capture
# of the named workload.  Reported only while the kernel sources hash to ``src``: any
# change to the kernel makes the figure stale, and then ``traffic`` is null.
KERNEL_SOURCES = ("tc_kernel.cuh", "tc_kernel.cu", "common.cuh", "sm100_ptx.cuh")
KERNEL_TRAFFIC = {
    "gqa_B2_Hq32_Hkv8_S4096_d128_causal_det:ordered": {
        "bytes": 621.7e6 + 285.2e6,
        "src": "a2d4e16f21418361",
        "profile": "profiles/bwd_tc_kernel_gqa_B2_S4096_det_traffic.md"},
}


def kernel_src_hash():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "head_attention_backward_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(key):
    t = KERNEL_TRAFFIC.get(key)
    if t is None or t["src"] != kernel_src_hash():
        return None, None
    return t["bytes"], t["profile"]


DQ_MODES = {"atomic": 0, "ordered": 1, "split": 2}
DQ_MODE_NAMES = {0: "atomic fp32 reductions", 1: "ordered fold (ascending KV tile)",
                 2: "split slices + fixed-order reduction"}


def dq_mode(wl):
    """attn_det_t value of a workload: False/True or an explicit mode."""
    return int(wl.deterministic)


def dq_mode_run(wl):
    """The dQ accumulation the library runs for the workload: the ordered fold
    is served by the split slices for fp32 inputs."""
    m = dq_mode(wl)
    if m == DQ_MODES["ordered"] and wl.dtype == torch.float32:
        return DQ_MODES["split"]
    return m


def config_of(wl):
    c = {"workload": wl.name, "batch": wl.batch, "nhead_q": wl.hq, "nhead_kv": wl.hkv,
         "seqlen": wl.sq, "d_qk": wl.d_qk, "d_v": wl.d_v, "mask": wl.mask,
         "window": [wl.left, wl.right], "deterministic": bool(wl.deterministic),
         "dq_mode": DQ_MODE_NAMES[dq_mode_run(wl)],
         "l2": "flushed (256 MB write) before every timed step"}
    if wl.group_mode:
        c["segments"] = len(wl.seqlens)
        c["total_tokens"] = wl.total
    return c


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        target = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", target], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].strip() not in ("", "[N/A]"))}


def cpu_sample(wl, x, groups, budget_s):
    """fp64 oracle backward on whole (batch, kv-head) groups of the workload;
    returns (mask-adjusted FLOPs done, seconds, description)."""
    from oracle import attn_ref as R
    g = wl.hq // wl.hkv
    per_pair = 2.0 * (3 * wl.d_qk + 2 * wl.d_v)
    pairs = FL.visible_pairs(wl.sq, wl.sk, wl.mask, wl.left, wl.right)
    done_flops, secs, n = 0.0, 0.0, 0
    for b, hk in groups:
        hs = slice(hk * g, (hk + 1) * g)
        q, k, v, do = (x["q"][b:b + 1, :, hs], x["k"][b:b + 1, :, hk:hk + 1], x["v"][b:b + 1, :, hk:hk + 1],
                       x["do"][b:b + 1, :, hs])
        kw = dict(mask=wl.mask, left=wl.left, right=wl.right)
        o, lse = R.attn_forward(q, k, v, wl.scale, **kw)
        t0 = time.perf_counter()
        R.attn_backward(q, k, v, o, do, lse, wl.scale, **kw)
        secs += time.perf_counter() - t0
        done_flops += per_pair * pairs * g
        n += 1
        if secs >= budget_s:
            break
    return done_flops, secs, f"{n} (batch, kv-head) group(s) x {g} query heads of {wl.name}, full S={wl.sq}"


def run_reference(args, wl):
    """The fp64 oracle timed on the host cores.  One step = the backward of one
    query head (with its kv head) of the workload at full sequence length; the
    forward that feeds it is computed once per head, outside the timed region."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import attn_ref as R
    x = wl.inputs()
    g = wl.hq // wl.hkv
    kw = dict(mask=wl.mask, left=wl.left, right=wl.right)
    per_head = 2.0 * (3 * wl.d_qk + 2 * wl.d_v) * FL.visible_pairs(wl.sq, wl.sk, wl.mask, wl.left, wl.right)
    fwd = {}
    secs = []
    for i in range(args.warmup + args.steps):
        h = i % wl.hq
        q, k, v, do = (x["q"][0:1, :, h:h + 1], x["k"][0:1, :, h // g:h // g + 1],
                       x["v"][0:1, :, h // g:h // g + 1], x["do"][0:1, :, h:h + 1])
        if h not in fwd:
            fwd[h] = R.attn_forward(q, k, v, wl.scale, **kw)
        o, lse = fwd[h]
        t0 = time.perf_counter()
        R.attn_backward(q, k, v, o, do, lse, wl.scale, **kw)
        if i >= args.warmup:
            secs.append(time.perf_counter() - t0)
    tot_s = sum(secs)
    value = per_head * len(secs) / tot_s / 1e12
    cores = torch.get_num_threads()
    desc = f"per step: the backward of one query head of {wl.name} (batch 0, full S={wl.sq}, dense fp64 scores)"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / len(secs),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": config_of(wl),
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ours(args, wl):
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from head_attention_backward_gb300 import build as BLD
    if rank == 0:
        BLD.build_library()
    if pg:
        pg.barrier()
    BLD.build_library()
    from head_attention_backward_gb300 import binding as B
    B.load()

    x = wl.inputs()
    d = {k: v.to(dev) for k, v in x.items()}
    cu = wl.cu_seqlens()
    cu_d = None if cu is None else cu.to(dev)
    cuk = wl.cu_seqlens_k()
    cuk_d = None if cuk is None else cuk.to(dev)
    kw = dict(scale=wl.scale, mask=wl.mask, left=wl.left, right=wl.right, cu_seqlens_q=cu_d,
              cu_seqlens_k=cuk_d, max_seqlen_q=wl.sq, max_seqlen_k=wl.sk)
    o, lse = B.attn_forward(d["q"], d["k"], d["v"], **kw)
    # the forward that made O and LSE, timed for the record (not part of a step):
    # the attn_fwd C-ABI call on prebuilt parameters, L2 flushed before each call
    # (the flush also keeps the GPU busy while the host enqueues the launch)
    fo, flse = torch.empty_like(o), torch.empty_like(lse)
    fo.copy_(o)
    flse.copy_(lse)
    pf = B.fwd_params(d["q"], d["k"], d["v"], fo, flse, **kw)
    fflush = torch.empty(256 * 2**20 // 4, dtype=torch.float32, device=dev)
    fstream = torch.cuda.current_stream(dev).cuda_stream
    fwd_ms = []
    for i in range(13):
        fflush.fill_(1.0)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        fst = B.attn_fwd(pf, fstream)
        f1.record()
        f1.synchronize()
        if fst != 0:
            raise RuntimeError(f"attn_fwd failed with status {fst}")
        if i >= 3:
            fwd_ms.append(f0.elapsed_time(f1))
    fwd_ms = sorted(fwd_ms)[len(fwd_ms) // 2]
    del fflush
    outs = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]))
    p = B.bwd_params(d["q"], d["k"], d["v"], o, d["do"], lse, *outs, deterministic=dq_mode(wl), **kw)
    nbytes = B.workspace_bytes(p)
    ws = B.alloc_workspace(nbytes, dev)
    flush = torch.empty(256 * 2**20 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    fl = FL.bwd_flops(wl)

    def step():
        flush.fill_(1.0)
        st, ms = B.attn_bwd_timed(p, ws.data_ptr(), nbytes, stream)
        if st != 0:
            raise B.AttnError(st, "attn_bwd_timed")
        return ms

    for _ in range(args.warmup):
        step()
    st, dev_status = B.attn_bwd_read_status(ws.data_ptr(), stream)
    if st != 0 or dev_status != 0:
        raise B.AttnError(dev_status or st, "device status after warm-up")
    clocks = ClockSampler(local)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    stage = [step() for _ in range(args.steps)]
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if pg:
        pg.barrier()
    clk = clocks.stop()
    step_ms = [s[3] for s in stage]
    main_ms = [s[1] for s in stage]
    ms_per_step = sum(step_ms) / len(step_ms)
    main_avg = sum(main_ms) / len(main_ms)
    ms_per_step, main_avg = max_over_ranks([ms_per_step, main_avg], pg, dev)

    # the pages' split-slice workspace on the same workload (same bits as the
    # ordered fold), timed beside it for reference
    split_leg = None
    if dq_mode_run(wl) == DQ_MODES["ordered"] and not args.no_split_leg:
        ps = B.bwd_params(d["q"], d["k"], d["v"], o, d["do"], lse, *outs, deterministic=DQ_MODES["split"], **kw)
        nb = B.workspace_bytes(ps)
        wss = B.alloc_workspace(nb, dev)
        sms = []
        for i in range(3 + min(args.steps, 20)):
            flush.fill_(1.0)
            st, ms = B.attn_bwd_timed(ps, wss.data_ptr(), nb, stream)
            if st != 0:
                raise B.AttnError(st, "attn_bwd_timed (split)")
            if i >= 3:
                sms.append(ms)
        del wss
        sp_ms = max_over_ranks([sum(m[3] for m in sms) / len(sms)], pg, dev)[0]
        split_leg = {"dq_mode": DQ_MODE_NAMES[DQ_MODES["split"]], "ms_per_step": sp_ms,
                     "value": job_throughput(world, fl, sp_ms), "steps": len(sms),
                     "step_stage_ms": [sum(m[k] for m in sms) / len(sms) for k in range(4)],
                     "workspace_bytes": nb}

    # end to end through the C ABI: pinned host inputs in, results back out
    e2e_avg, h2d, d2h, e2e_chunks = float("nan"), 0, 0, 0
    if not args.no_e2e:
        host = {k: v.to(dev).cpu().pin_memory() for k, v in (("q", d["q"]), ("k", d["k"]), ("v", d["v"]),
                                                               ("o", o), ("do", d["do"]), ("lse", lse))}
        host_out = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in outs)
        e2e_ms = []
        # attn_bwd_host: chunk c's copies overlap its neighbours' compute
        h = B.host_tensors(host["q"], host["k"], host["v"], host["o"], host["do"], host["lse"], *host_out)
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        chunks = e2e_chunks = args.e2e_chunks if args.e2e_chunks > 0 else max(1, min(wl.batch, 4))
        for i in range(args.warmup + args.steps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            rc = B.attn_bwd_host(p, h, ws.data_ptr(), nbytes, stream, s_in.cuda_stream, s_out.cuda_stream, chunks)
            if rc != 0:
                raise B.AttnError(rc, "attn_bwd_host")
            e1.record()
            e1.synchronize()
            if i >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        e2e_avg = max_over_ranks([sum(e2e_ms) / len(e2e_ms)], pg, dev)[0]

    peak_tf, peak_hbm, peak_src = peaks()
    traffic, traffic_src = measured_traffic(f"{wl.name}:{[k for k, v in DQ_MODES.items() if v == dq_mode(wl)][0]}")
    value = job_throughput(world, fl, ms_per_step)
    achieved = fl / (main_avg * 1e-3) / 1e12
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == torch.bfloat16 else str(wl.dtype),
        "data": "synthetic", "config": config_of(wl),
        "pct_of_peak": 100.0 * value / world / peak_tf,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": traffic, "traffic_source": traffic_src,
                     "kernel": "bwd_tc_kernel",
                     "peak_source": f"{peak_src} bf16 burst", "kernel_ms": main_avg,
                     "step_stage_ms": [sum(s[i] for s in stage) / len(stage) for i in range(4)]},
        "e2e": None if args.no_e2e else {"value": job_throughput(world, fl, e2e_avg), "unit": "TFLOP/s",
                                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                         "ms_per_step": e2e_avg, "api": "attn_bwd_host", "chunks": e2e_chunks},
        # the library's own kernels per step: preprocess, main, reduce/convert,
        # plus the scheduler in group mode (batch mode schedules in the preprocess)
        "gpu_launches": (4 if wl.group_mode else 3) * args.steps,
        "forward": {"kernel": "fwd_tc_kernel" if wl.dtype != torch.float32 else "fwd_kernel",
                    "ms": fwd_ms, "TFLOP/s": fl * (wl.d_qk + wl.d_v) / (3 * wl.d_qk + 2 * wl.d_v) / fwd_ms / 1e9,
                    "note": "median of 10 attn_fwd C-ABI calls on prebuilt parameters, L2 flushed before each; not part of the timed step"},
        "split_slices": split_leg,
        "clocks": clk,
        "workspace_bytes": nbytes,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        groups = [(b, hk) for b in range(wl.batch) for hk in range(wl.hkv)]
        f, s, desc = cpu_sample(wl, x, groups, args.cpu_budget)
        out["cpu_baseline"] = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(),
                               "kind": "oracle", "sample": desc + f" ({s:.1f} s of fp64 CPU work, dense scores)"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_causal_det", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="chunks of the end-to-end leg (0: min(batch, 4) runs of batch entries)")
    ap.add_argument("--batch", type=int, default=0, help="override the batch of a batch-mode workload")
    ap.add_argument("--atomic", action="store_true", help="same as --dq-mode atomic")
    ap.add_argument("--dq-mode", choices=sorted(DQ_MODES), default=None,
                    help="dQ accumulation: ordered fold, split slices or fp32 atomics (default: the workload's)")
    ap.add_argument("--no-split-leg", action="store_true",
                    help="skip timing the split-slice path beside the ordered fold")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]()
    if args.batch and not wl.group_mode:
        wl.batch = args.batch
        wl.name += f"_batch{args.batch}"
    if args.atomic:
        args.dq_mode = "atomic"
    if args.dq_mode is not None:
        wl.deterministic = DQ_MODES[args.dq_mode]
        if args.dq_mode == "atomic":
            wl.name += "_atomic"
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
