"""Benchmark of the gated causal prefill path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu] [--no-sweep]

Default workload: one Llama-3.1-8B attention layer at L = 131072 (32 query
heads, 8 KV heads, d = 128, Bq = Bk = 128) with a 256-token sink and 64
needle blocks per KV head; thresholds calibrated by bsfa_calibrate on four
seeded 64K inputs for budgets k = 32, 128, 512.  One step = the three budget
slices run back to back.  Inputs (Q 1 GiB, K and V 256 MiB each) exceed the
129 MB L2, so no flush is needed between iterations.

Prints ONE JSON line (rank 0).  value = effective TFLOP/s over the step,
effective FLOPs = 2*Bq*Bk*d * (visible blocks + kept blocks).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("prefill attention ms/layer & effective TFLOPS (frac of bf16 peak) at 128K vs "
          "skip rate")
UNIT = "TFLOP/s (effective)"


# The kernel the timed step runs (the default schedule for gated 128 x 128
# calls) and its own sources: an ncu record stays valid while these are
# unchanged (host-side code, such as argument checks, does not affect it).
ROOFLINE_KERNEL = "bsfa_xs_kernel"
KERNEL_SOURCES = ["block_sparse_gated_gb300/csrc/bsfa_xs.cuh",
                  "block_sparse_gated_gb300/csrc/bsfa_fwd.cuh",
                  "block_sparse_gated_gb300/csrc/ptx.cuh",
                  "block_sparse_gated_gb300/csrc/inst_xs.cuh"]


def code_digest(paths=KERNEL_SOURCES):
    """sha256 of the given sources with C/C++ comments and all whitespace
    removed: it changes when the code changes, not when a comment does."""
    import hashlib
    import re
    h = hashlib.sha256()
    for p in paths:
        text = open(os.path.join(ROOT, p)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()


def _recorded_traffic(workload):
    """Mean DRAM bytes per launch of the prefill kernel from the committed ncu
    record, or None when the kernel code changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{ROOFLINE_KERNEL}_dram_{workload}.json")
    try:
        rec = json.load(open(path))
        if rec["sources"] != KERNEL_SOURCES or code_digest() != rec["code_sha256"]:
            return None
        return float(rec["mean_bytes_per_launch"])
    except Exception:
        return None


def _recorded_ncu(workload="llama8b-L32768"):
    """Tensor-pipe utilisation and DRAM GB/s from the committed full ncu
    capture of the prefill kernel, or None when the kernel code changed since
    it was taken."""
    path = os.path.join(ROOT, "profiles", f"{ROOFLINE_KERNEL}_full_{workload}.json")
    try:
        rec = json.load(open(path))
        if rec["sources"] != KERNEL_SOURCES or code_digest() != rec["code_sha256"]:
            return None
        return {"workload": rec["workload"], "kernel": rec["kernel"],
                "tensor_pipe_active_pct": rec["tensor_pipe_active_pct_of_elapsed"],
                "dram_gbps": rec["dram_gbps"],
                "dram_pct_of_peak": rec["dram_throughput_pct_of_peak"],
                "source": os.path.relpath(path, ROOT)}
    except Exception:
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, val in zip(names, f[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload
def _cfg(name):
    from block_sparse_gated_gb300 import workloads as wl
    return wl.WORKLOADS[name]


def build_workload(name, device):
    """Inputs on the device and the calibrated threshold slices (GPU path)."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    from block_sparse_gated_gb300 import workloads as wl
    cfg = _cfg(name)
    Hq, Hkv, d, Bq, Bk = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bq"], cfg["Bk"]
    cal = []
    for n in range(cfg["n_cal"]):
        x = wl.layer_inputs(Hq, Hkv, cfg["cal_L"], d, wl.cal_seed(cfg["index"], n), device,
                            with_v=False, sink_tokens=cfg["sink_tokens"],
                            needles=cfg["cal_needles"], block=Bk)
        cal.append((x.q, x.k))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    T = bsfa.calibrate([c[0] for c in cal], [c[1] for c in cal], cfg["ks"], block_q=Bq, block_k=Bk)
    ev1.record()
    torch.cuda.synchronize()
    cal_ms = ev0.elapsed_time(ev1)
    nq_cal = T.shape[2]
    cal_flops = cfg["n_cal"] * Hq * 2.0 * Bq * Bk * d * (nq_cal * (nq_cal + 1) / 2)
    del cal
    x = wl.layer_inputs(Hq, Hkv, cfg["L"], d, wl.eval_seed(cfg["index"]), device,
                        sink_tokens=cfg["sink_tokens"], needles=cfg["needles"], block=Bk)
    torch.cuda.synchronize()
    return {"cfg": cfg, "q": x.q, "k": x.k, "v": x.v, "T": T, "cal_ms": cal_ms,
            "cal_tflops": cal_flops / (cal_ms * 1e-3) / 1e12,
            "gen_s": time.perf_counter() - t0}


def effective_flops(counts, Bq, Bk, d):
    kept_c, cand, diag = counts
    return 2.0 * Bq * Bk * d * ((cand + diag) + (kept_c + diag))


# ----------------------------------------------------------------- our arm
def aggregate_step(ms_step, step_flops, world, device=None):
    """Whole-job figures of a weak-scaling run: every rank runs one replica of
    the step, the step time is the maximum over ranks, and the value is the
    FLOPs of all ranks over that time (TFLOP/s).  Returns (ms, value)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())
    return ms_step, world * step_flops / (ms_step * 1e-3) / 1e12


def aggregate_shards(ms_step, step_flops, world, device=None):
    """Whole-job figures of a head-sharded run: each rank computes its own KV
    heads (and their query heads) of the same layer, the step time is the
    maximum over ranks, and the value is the FLOPs summed over ranks over
    that time (TFLOP/s).  Returns (ms, value, total FLOPs)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
        f = torch.tensor([float(step_flops)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(f, op=dist.ReduceOp.SUM)
        ms_step, step_flops = float(t.item()), float(f.item())
    return ms_step, step_flops / (ms_step * 1e-3) / 1e12, step_flops


def _check_device(bsfa, what):
    """Every kernel wait is bounded; one that ran out sets the device error
    word and the kernel returns early, so its timing and outputs mean
    nothing.  Refuse to report them."""
    code = bsfa.api.device_error()
    if code != 0:
        raise RuntimeError(f"{what}: a device-side wait ran out (site {code:#x}); "
                           "no number is reported")


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import block_sparse_gated_gb300 as bsfa
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peak_burst, peak_sust, peak_kind = _peaks()
    W = build_workload(args.workload, dev)
    cfg = W["cfg"]
    Hq, d, Bq, Bk, L = cfg["Hq"], cfg["d"], cfg["Bq"], cfg["Bk"], cfg["L"]
    q, k, v, T = W["q"][None], W["k"][None], W["v"][None], W["T"]
    sharded = args.shard == "heads"
    if sharded:
        from block_sparse_gated_gb300.shard import head_shard, shard_tensors
        sh = head_shard(Hq, cfg["Hkv"], rank, world)
        q, k, v, T = (t.contiguous() for t in shard_tensors(sh, q, k, v, T))
        Hq = sh.num_heads_q
    ks = cfg["ks"]
    slices = [T[i].contiguous() for i in range(len(ks))]
    outs = [torch.empty_like(q) for _ in ks]
    counts = [torch.zeros(3, dtype=torch.int64, device=dev) for _ in ks]
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(i):
        bsfa.prefill(q, k, v, block_q=Bq, block_k=Bk, mode="threshold", thresholds=slices[i],
                     out=outs[i], workspace=ws, stream=stream)

    # counts: one untimed pass with counters on
    for i in range(len(ks)):
        r = bsfa.prefill(q, k, v, block_q=Bq, block_k=Bk, mode="threshold",
                         thresholds=slices[i], out=outs[i], workspace=ws, return_counts=True)
        counts[i] = r["counts"]
    torch.cuda.synchronize()
    cnts = [c.cpu().tolist() for c in counts]
    flops = [effective_flops(c, Bq, Bk, d) for c in cnts]

    starts = [[torch.cuda.Event(enable_timing=True) for _ in ks] for _ in range(args.steps)]
    ends = [[torch.cuda.Event(enable_timing=True) for _ in ks] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        # Warm up after the sampler has started, so the GPU does not sit idle
        # (and drop its clocks) between the warm-up and the timed steps.
        for _ in range(args.warmup):
            for i in range(len(ks)):
                call(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for s in range(args.steps):
            for i in range(len(ks)):
                starts[s][i].record(stream)
                call(i)
                ends[s][i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = clk.summary()
    _check_device(bsfa, "timed step")
    total_ms = t_start.elapsed_time(t_end)
    step_flops = sum(flops)
    if sharded:
        ms_step, value, _ = aggregate_shards(total_ms / args.steps, step_flops, world, dev)
    else:
        ms_step, value = aggregate_step(total_ms / args.steps, step_flops, world, dev)
    per_slice_ms = [statistics.mean(starts[s][i].elapsed_time(ends[s][i]) for s in range(args.steps))
                    for i in range(len(ks))]
    launch_achieved = sum(flops) / (sum(per_slice_ms) * 1e-3) / 1e12
    slices_out = []
    for i, kk in enumerate(ks):
        kc, cand, diag = cnts[i]
        tf = flops[i] / (per_slice_ms[i] * 1e-3) / 1e12
        slices_out.append({
            "k": kk, "ms_per_layer": round(per_slice_ms[i], 3),
            "skip_rate": round(1.0 - kc / cand, 4) if cand else 0.0,
            "density": round((kc + diag) / (cand + diag), 4),
            "effective_tflops": round(tf, 1),
            "frac_of_burst_peak": round(tf / peak_burst, 4),
            "frac_of_sustained_peak": round(tf / peak_sust, 4)})

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "strong" if sharded else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; Llama-3.1-8B attention shapes; no dataset)",
        "config": {"workload": args.workload, "Hq": Hq, "Hkv": cfg["Hkv"], "d": d, "L": L,
                   "Bq": Bq, "Bk": Bk, "budgets_k": ks, "calibration": f"{cfg['n_cal']} x "
                   f"{cfg['cal_L']} tokens",
                   "schedule": bsfa.api.resolve_schedule("auto", mode="threshold", block_q=Bq,
                                                         block_k=Bk),
                   "l2": f"inputs larger than L2 (Q {q.numel() * 2 / 2**20:.0f} MiB, K and V "
                         f"{k.numel() * 2 / 2**20:.0f} MiB each); no flush",
                   "parallelism": (f"heads x{world} (rank 0: KV heads "
                                   f"{sh.kv_heads.start}-{sh.kv_heads.stop - 1}, slices below are "
                                   f"rank 0's)" if sharded else f"replica x{world}")},
        "slices": slices_out,
        "roofline": {"bound": "tensor", "achieved": round(launch_achieved, 1),
                     "peak": peak_sust, "unit": "TFLOP/s",
                     "frac": round(launch_achieved / peak_sust, 4),
                     "peak_kind": f"{peak_kind} bf16 sustained (kernel timed inside a long step)",
                     "frac_of_burst": round(launch_achieved / peak_burst, 4),
                     "traffic": _recorded_traffic(args.workload),
                     "traffic_unit": "bytes per launch (ncu dram read + write)",
                     "ncu": _recorded_ncu()},
        "clocks": clocks,
        "gpu_launches": 2 * len(ks) * args.steps,
        "calibrate": {"ms": round(W["cal_ms"], 3), "samples": cfg["n_cal"],
                      "tflops_qk": round(W["cal_tflops"], 1)},
    }

    if not args.no_sweep and rank == 0 and not sharded:
        result["paged_kv"] = paged_leg(q, k, v, slices, ks, outs, Bq, Bk, dev)
        result["mean_correction"] = mean_correction_leg(q, k, v, slices, ks, Bq, Bk, dev)
        result["lambda_sweep"] = lambda_sweep(dev, args)
        result["llama8b_L32768"] = llama_32k_leg(dev)
        result["varlen_8seq_32layer"] = varlen_32layer_leg(dev)
        result["tile_128x224"] = tile224_leg(dev)
    if not args.no_e2e and not sharded:
        result["e2e"] = e2e(q, k, v, slices, flops, Bq, Bk, args, dev)
    _check_device(bsfa, "bench legs")
    if not args.no_cpu and rank == 0 and world == 1 and not sharded:
        result["cpu_baseline"] = cpu_baseline(args.workload, W, cnts)
    if rank == 0:
        print(json.dumps(result), flush=True)


def paged_leg(q, k, v, slices, ks, outs, Bq, Bk, dev, page=256, reps=3):
    """The k=128 slice of the same layer with K and V read from page pools
    ([pages, 256, Hkv, d], pages in a seeded random order) through a block
    table, against the contiguous call; the outputs must be identical."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    i = ks.index(128) if 128 in ks else 0
    L = k.shape[2]
    n_pages = (L + page - 1) // page
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(5)).to(dev)

    def pool(t):
        pad = n_pages * page - L
        x = torch.nn.functional.pad(t[0].transpose(0, 1), (0, 0, 0, 0, 0, pad))
        x = x.reshape(n_pages, page, t.shape[1], t.shape[3])
        out = torch.empty_like(x)
        out[perm] = x
        return out

    kp, vp = pool(k), pool(v)
    table = perm.to(torch.int32)[None].contiguous()
    ref = outs[i]
    got = torch.empty_like(ref)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    bsfa.prefill(q, k, v, block_q=Bq, block_k=Bk, mode="threshold", thresholds=slices[i],
                 out=ref, workspace=ws)
    bsfa.prefill(q, kp, vp, block_q=Bq, block_k=Bk, mode="threshold", thresholds=slices[i],
                 out=got, workspace=ws, block_table=table)
    torch.cuda.synchronize()
    same = bool(torch.equal(got, ref))
    ms_c = _timed(lambda: bsfa.prefill(q, k, v, block_q=Bq, block_k=Bk, mode="threshold",
                                       thresholds=slices[i], out=ref, workspace=ws), reps)
    ms_p = _timed(lambda: bsfa.prefill(q, kp, vp, block_q=Bq, block_k=Bk, mode="threshold",
                                       thresholds=slices[i], out=got, workspace=ws,
                                       block_table=table), reps)
    del kp, vp
    return {"k": ks[i], "page_size": page, "pages": n_pages, "order": "seeded random permutation",
            "ms_contiguous": round(ms_c, 3), "ms_paged": round(ms_p, 3),
            "paged_over_contiguous": round(ms_p / ms_c, 4), "outputs_identical": same}


def mean_correction_leg(q, k, v, slices, ks, Bq, Bk, dev, reps=3):
    """Cost of the mean-correction option on the k=128 slice: the same gate
    (identical bitmap), plus the block-mean pass and one correction tile per
    128 candidate blocks of every query tile.  Both kernels carry the option;
    each is timed with and without it, and "default" names the one that
    schedule="auto" takes for a corrected call."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    i = ks.index(128) if 128 in ks else 0
    out = torch.empty_like(q)
    kw = dict(block_q=Bq, block_k=Bk, mode="threshold", thresholds=slices[i], out=out)
    need = bsfa.api.prefill_workspace_bytes(q, k, v, mean_correction=True, **kw)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    res = {"k": ks[i],
           "default": bsfa.api.resolve_schedule("auto", mode="threshold", block_q=Bq,
                                                block_k=Bk, mean_correction=True),
           "workspace_bytes": int(need)}
    for sched in ("pipelined", "paired"):
        kw["schedule"] = sched
        a = bsfa.prefill(q, k, v, return_bitmap=True, workspace=ws, **kw)["bitmap"].clone()
        b = bsfa.prefill(q, k, v, return_bitmap=True, workspace=ws, mean_correction=True,
                         **kw)["bitmap"]
        torch.cuda.synchronize()
        same = bool(torch.equal(a, b))
        del a, b
        ms_plain = _timed(lambda: bsfa.prefill(q, k, v, workspace=ws, **kw), reps)
        ms_corr = _timed(lambda: bsfa.prefill(q, k, v, workspace=ws, mean_correction=True,
                                              **kw), reps)
        res[sched] = {"ms_plain": round(ms_plain, 3), "ms_corrected": round(ms_corr, 3),
                      "corrected_over_plain": round(ms_corr / ms_plain, 4),
                      "bitmap_identical": same}
    return res


def e2e(q, k, v, slices, flops, Bq, Bk, args, dev):
    """Same metric through the public API with host buffers.  Every step
    copies that step's pinned Q/K/V host->device, runs the three budget
    slices and copies the three outputs device->host.  Copies run on a copy
    stream and overlap the previous/next step's attention on the compute
    stream (double-buffered device inputs and outputs, ordered by events;
    uploads and downloads on separate streams),
    as a serving loop would; the timed region spans all steps end to end."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    n = max(2, args.steps)  # the device-timed step count; the first upload and the last
    # download of the timed region overlap nothing, so fewer steps would weigh them more
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = [[torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in slices] for _ in range(2)]
    din = [[torch.empty_like(t) for t in (q, k, v)] for _ in range(2)]
    dout = [[torch.empty_like(q) for _ in slices] for _ in range(2)]
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev(), ev()]
    in_free = [ev(), ev()]
    out_ready = [[ev() for _ in slices] for _ in range(2)]
    out_free = [[ev() for _ in slices] for _ in range(2)]

    def run(steps):
        for st in range(steps):
            b = st % 2
            with torch.cuda.stream(h2d_s):
                if st >= 2:
                    h2d_s.wait_event(in_free[b])
                for dst, src in zip(din[b], (qh, kh, vh)):
                    dst.copy_(src, non_blocking=True)
                in_ready[b].record(h2d_s)
            comp.wait_event(in_ready[b])
            for i, T in enumerate(slices):
                if st >= 2:
                    comp.wait_event(out_free[b][i])
                bsfa.prefill(din[b][0], din[b][1], din[b][2], block_q=Bq, block_k=Bk,
                             mode="threshold", thresholds=T, out=dout[b][i], workspace=ws,
                             stream=comp)
                out_ready[b][i].record(comp)
            in_free[b].record(comp)
            with torch.cuda.stream(d2h_s):
                for i in range(len(slices)):
                    d2h_s.wait_event(out_ready[b][i])
                    oh[b][i].copy_(dout[b][i], non_blocking=True)
                    out_free[b][i].record(d2h_s)

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(n)
    comp.wait_stream(h2d_s)
    comp.wait_stream(d2h_s)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = sum(t.numel() * t.element_size() for t in oh[0])
    return {"value": round(sum(flops) / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": n, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "how": "pinned host buffers; upload and download streams overlapped with compute"}


def lambda_sweep(dev, args):
    """lambda gate at 64K: time vs dialled skip rate, plus the same kernel with
    the gate compiled out (0-skip overhead), and the A/B against loading V for
    skipped tiles too (``v_always``: same results, V read for every tile)."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    from block_sparse_gated_gb300 import workloads as wl
    cfg = _cfg("lambda-sweep-L65536")
    Hq, Hkv, d, L, B = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["L"], cfg["Bk"]
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    reps = 3
    rows = []

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for n, r in enumerate(cfg["skip_rates"]):
        x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"], n), dev, skip_rate=r, block=B)
        q, k, v = x.q[None], x.k[None], x.v[None]
        out = torch.empty_like(q)
        ll = cfg["log_lambda"] if r > 0 else -1e30  # 0%: evaluated gate keeping every block
        res = bsfa.prefill(q, k, v, mode="lambda", log_lambda=ll, out=out, workspace=ws,
                           return_counts=True)
        torch.cuda.synchronize()
        kc, cand, diag = res["counts"].cpu().tolist()
        ms = timed(lambda: bsfa.prefill(q, k, v, mode="lambda", log_lambda=ll, out=out,
                                        workspace=ws))
        row = {"target_skip": r, "log_lambda": ll,
               "measured_skip": round(1 - kc / cand, 4), "ms": round(ms, 3),
               "effective_tflops": round(effective_flops((kc, cand, diag), B, B, d) /
                                         (ms * 1e-3) / 1e12, 1),
               "ms_v_always": round(timed(lambda: bsfa.prefill(
                   q, k, v, mode="lambda", log_lambda=ll, out=out, workspace=ws,
                   v_always=True)), 3),
               "ms_paired": round(timed(lambda: bsfa.prefill(
                   q, k, v, mode="lambda", log_lambda=ll, out=out, workspace=ws,
                   schedule="paired")), 3)}
        if r == 0:
            # The gate evaluated (threshold and ln(lambda) -1e30: every block
            # kept after the vote), and -inf, which the kernels recognise as
            # keep-everything (no vote in the paired kernel, no exact running
            # max in the one-head kernel); each in both schedules.
            thr = torch.full((Hq, 1), -1e30, device=dev)
            thr_inf = torch.full((Hq, 1), -math.inf, device=dev)
            for sch, sfx in (("auto", ""), ("paired", "_paired")):
                row["ms_threshold_keep_all" + sfx] = round(timed(lambda: bsfa.prefill(
                    q, k, v, mode="threshold", thresholds=thr, out=out, workspace=ws,
                    schedule=sch)), 3)
                row["ms_threshold_minus_inf" + sfx] = round(timed(lambda: bsfa.prefill(
                    q, k, v, mode="threshold", thresholds=thr_inf, out=out, workspace=ws,
                    schedule=sch)), 3)
                row["ms_lambda_minus_inf" + sfx] = round(timed(lambda: bsfa.prefill(
                    q, k, v, mode="lambda", log_lambda=-math.inf, out=out, workspace=ws,
                    schedule=sch)), 3)
            row["ms_gate_compiled_out"] = round(timed(lambda: bsfa.prefill(
                q, k, v, mode="none", out=out, workspace=ws, schedule="paired")), 3)
            row["ms_gate_compiled_out_pipelined"] = round(timed(lambda: bsfa.prefill(
                q, k, v, mode="none", out=out, workspace=ws, schedule="pipelined")), 3)
        rows.append(row)
        del x, q, k, v, out
    r0 = rows[0]
    # Against the faster of the two gate-compiled-out kernels.
    base = min(r0["ms_gate_compiled_out"], r0["ms_gate_compiled_out_pipelined"])
    times = [r_["ms"] for r_ in rows]

    def ovh(key):
        return round(r0[key] / base - 1, 4)
    return {"workload": "lambda-sweep-L65536", "rows": rows,
            "gate_compiled_out_ms": round(base, 3),
            "zero_skip_overhead_lambda": round(r0["ms"] / base - 1, 4),
            "zero_skip_overhead_threshold": ovh("ms_threshold_keep_all"),
            "zero_skip_overhead_minus_inf": {
                "threshold": ovh("ms_threshold_minus_inf"),
                "lambda": ovh("ms_lambda_minus_inf"),
                "note": "a -inf threshold row (calibration gives one to query blocks with fewer "
                        "than k candidates) or ln(lambda) = -inf keeps every block"},
            # Against the same (default, one-head) kernel with the gate compiled out.
            "zero_skip_overhead_same_kernel": {
                "gate_compiled_out_ms": r0["ms_gate_compiled_out_pipelined"],
                "threshold": round(r0["ms_threshold_keep_all"] /
                                   r0["ms_gate_compiled_out_pipelined"] - 1, 4),
                "lambda": round(r0["ms"] / r0["ms_gate_compiled_out_pipelined"] - 1, 4),
                "threshold_minus_inf": round(r0["ms_threshold_minus_inf"] /
                                             r0["ms_gate_compiled_out_pipelined"] - 1, 4),
                "lambda_minus_inf": round(r0["ms_lambda_minus_inf"] /
                                          r0["ms_gate_compiled_out_pipelined"] - 1, 4)},
            "zero_skip_overhead_paired": {
                "lambda": round(r0["ms_paired"] / base - 1, 4),
                "threshold": ovh("ms_threshold_keep_all_paired"),
                "threshold_minus_inf": ovh("ms_threshold_minus_inf_paired"),
                "lambda_minus_inf": ovh("ms_lambda_minus_inf_paired")},
            "zero_skip_gate": "evaluated: threshold and ln(lambda) of -1e30 keep every block "
                              "after the vote; overheads against the faster gate-compiled-out "
                              "kernel",
            "skip90_speedup_over_gate_compiled_out": round(base / rows[-1]["ms"], 3),
            "monotonic": all(a > b for a, b in zip(times, times[1:])),
            "v_always_over_gated_v": [round(r_["ms_v_always"] / r_["ms"], 4) for r_ in rows],
            "pipelined_over_paired": [round(r_["ms"] / r_["ms_paired"], 4) for r_ in rows],
            "schedules": "ms*: the default schedule (auto: one query head per CTA, Q.K^T issued "
                         "ahead of P.V by a warp of its own); *_paired: two query heads of a GQA "
                         "group per CTA sharing each K/V tile; gate compiled out: paired, and "
                         "*_pipelined the one-head kernel"}


def tile224_leg(dev, reps=3):
    """The H100 port's 128 x 224 tile on the 64K lambda-sweep layer shape (32
    query heads, 8 KV heads, d = 128): the lambda gate at dialled 0% and 50%
    skip (key scale tiers drawn per 224-key block), and the gate compiled out.
    Effective FLOPs count 2 * 128 * 224 * d per visible tile and again per
    kept tile."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    from block_sparse_gated_gb300 import workloads as wl
    cfg = _cfg("lambda-sweep-L65536")
    Hq, Hkv, d, L = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["L"]
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    rows = []
    for n, r in enumerate((0.0, 0.5)):
        x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"], 20 + n), dev, skip_rate=r,
                            block=224)
        q, k, v = x.q[None], x.k[None], x.v[None]
        out = torch.empty_like(q)
        ll = cfg["log_lambda"] if r > 0 else -1e30  # 0%: evaluated gate keeping every block
        kw = dict(block_q=128, block_k=224, out=out, workspace=ws)
        res = bsfa.prefill(q, k, v, mode="lambda", log_lambda=ll, return_counts=True, **kw)
        torch.cuda.synchronize()
        kc, cand, diag = res["counts"].cpu().tolist()
        ms = _timed(lambda: bsfa.prefill(q, k, v, mode="lambda", log_lambda=ll, **kw), reps)
        row = {"target_skip": r, "measured_skip": round(1 - kc / cand, 4), "ms": round(ms, 3),
               "effective_tflops": round(2.0 * 128 * 224 * d * (cand + diag + kc + diag) /
                                         (ms * 1e-3) / 1e12, 1)}
        if r == 0:
            row["ms_gate_compiled_out"] = round(_timed(lambda: bsfa.prefill(
                q, k, v, mode="none", **kw), reps), 3)
        rows.append(row)
        del x, q, k, v, out
    return {"workload": "lambda-sweep-L65536 shape, Bq=128 Bk=224", "rows": rows,
            "kernel": "single-head kernel, one 224-column score buffer"}


def _timed(fn, reps):
    import torch
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def llama_32k_leg(dev, reps=5):
    """The 32K layer: thresholds calibrated on 4 x 32K samples, k = 64."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    W = build_workload("llama8b-L32768", dev)
    cfg = W["cfg"]
    q, k, v, T = W["q"][None], W["k"][None], W["v"][None], W["T"][0].contiguous()
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    r = bsfa.prefill(q, k, v, mode="threshold", thresholds=T, out=out, workspace=ws,
                     return_counts=True)
    torch.cuda.synchronize()
    kc, cand, diag = r["counts"].cpu().tolist()
    ms = _timed(lambda: bsfa.prefill(q, k, v, mode="threshold", thresholds=T, out=out,
                                     workspace=ws), reps)
    fl = effective_flops((kc, cand, diag), cfg["Bq"], cfg["Bk"], cfg["d"])
    return {"workload": "llama8b-L32768", "k": cfg["ks"][0], "ms_per_layer": round(ms, 3),
            "skip_rate": round(1 - kc / cand, 4),
            "effective_tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "calibrate_ms": round(W["cal_ms"], 3)}


def varlen_32layer_leg(dev):
    """8 sequences (4K..64K) packed with cu_seqlens; one threshold table per
    layer (k = 128, 4 x 64K calibration samples per layer); the 32 layers'
    slices run back to back over the packed batch (per-layer time = total / 32)."""
    import torch

    import block_sparse_gated_gb300 as bsfa
    from block_sparse_gated_gb300 import workloads as wl
    cfg = wl.WORKLOADS["varlen-8seq-32layer"]
    Hq, Hkv, d, B = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bk"]
    tables = []
    t_cal = 0.0
    for layer in range(cfg["layers"]):
        cal = [wl.layer_inputs(Hq, Hkv, cfg["cal_L"], d, wl.cal_seed(cfg["index"], n, layer), dev,
                               with_v=False, sink_tokens=cfg["sink_tokens"],
                               needles=cfg["cal_needles"], block=B) for n in range(cfg["n_cal"])]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        T = bsfa.calibrate([c.q for c in cal], [c.k for c in cal], cfg["ks"], block_q=B,
                           block_k=B)
        e1.record()
        torch.cuda.synchronize()
        t_cal += e0.elapsed_time(e1)
        tables.append(T[0].contiguous())
        del cal
    lens = cfg["lens"]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, wl.eval_seed(cfg["index"], n), dev,
                             sink_tokens=cfg["sink_tokens"],
                             needles=max(1, round(cfg["needles_per_64k"] * Ln / 65536)), block=B)
             for n, Ln in enumerate(lens)]
    q, cu = wl.pack_varlen([p_.q for p_ in parts])
    k, _ = wl.pack_varlen([p_.k for p_ in parts])
    v, _ = wl.pack_varlen([p_.v for p_ in parts])
    del parts
    cu = cu.to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    tot = [0, 0, 0]
    for T in tables:
        r = bsfa.prefill(q, k, v, cu_seqlens=cu, max_seqlen=max(lens), mode="threshold",
                         thresholds=T, out=out, workspace=ws, return_counts=True)
        torch.cuda.synchronize()
        tot = [a + b for a, b in zip(tot, r["counts"].cpu().tolist())]

    def all_layers():
        for T in tables:
            bsfa.prefill(q, k, v, cu_seqlens=cu, max_seqlen=max(lens), mode="threshold",
                         thresholds=T, out=out, workspace=ws)

    ms = _timed(all_layers, 2)
    fl = effective_flops(tot, B, B, d)
    return {"workload": "varlen-8seq-32layer", "tokens": int(sum(lens)), "layers": len(tables),
            "ms_per_layer": round(ms / len(tables), 3), "skip_rate": round(1 - tot[0] / tot[1], 4),
            "effective_tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "calibrate_ms_per_layer": round(t_cal / len(tables), 3)}


# --------------------------------------------------------------- CPU oracle
def oracle_sample(q_heads, k_heads, v_heads, heads, T_rows, blocks, Bq, Bk, sigma):
    """Time the oracle on sampled (head, query block) units.  Returns
    (effective FLOPs, seconds, n_blocks)."""
    from oracle import bsfa_oracle as orc
    d = q_heads[heads[0]].shape[1]
    F = 2.0 * Bq * Bk * d
    fl, t0 = 0.0, time.perf_counter()
    for h, i in blocks:
        r = orc.query_block(q_heads[h], k_heads[h], v_heads[h], i, Bq=Bq, Bk=Bk, sigma=sigma,
                            mode="threshold", T_hi=T_rows[(h, i)])
        fl += F * (len(r["keep"]) + sum(r["keep"].values()))
    return fl, time.perf_counter() - t0, len(blocks)


def _sample_blocks(n_q, nT, heads, per_head, seed):
    import random
    rnd = random.Random(seed)
    out = []
    for h in heads:
        fixed = sorted({0, nT - 1, min(nT, n_q - 1), n_q - 1})
        extra = rnd.sample(range(n_q), per_head)
        out += [(h, i) for i in sorted(set(fixed + extra))]
    return out


def _oracle_inputs(name, W=None, heads=(0, 9, 17, 30)):
    """fp64 host copies of the sampled heads (and their KV heads), and oracle
    thresholds for the sampled rows computed from the calibration recipe."""
    import numpy as np
    import torch

    from block_sparse_gated_gb300 import workloads as wl
    from oracle import bsfa_oracle as orc
    cfg = _cfg(name)
    Hq, Hkv, d, Bq, Bk = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bq"], cfg["Bk"]
    g = Hq // Hkv
    dev = W["q"].device if W is not None else "cpu"
    if W is None:
        # Host-only run: one KV-head group of the layer (g query heads over one
        # KV head); the per-block work of a (head, query block) is unchanged.
        cfg = dict(cfg, Hq=g, Hkv=1)
        Hq, Hkv = g, 1
        heads = tuple(range(g))
        x = wl.layer_inputs(Hq, Hkv, cfg["L"], d, wl.eval_seed(cfg["index"]), "cpu",
                            sink_tokens=cfg["sink_tokens"], needles=cfg["needles"], block=Bk)
        q, k, v = x.q, x.k, x.v
    else:
        q, k, v = W["q"], W["k"], W["v"]
    qh = {h: q[h].to("cpu", torch.float64).numpy() for h in heads}
    kh = {h: k[h // g].to("cpu", torch.float64).numpy() for h in heads}
    vh = {h: v[h // g].to("cpu", torch.float64).numpy() for h in heads}
    return cfg, qh, kh, vh


def _oracle_thresholds(cfg, heads, blocks, device):
    """Oracle calibration restricted to the table entries the sampled blocks
    read (k = the smallest budget), from the calibration recipe's inputs."""
    import numpy as np
    import torch

    from block_sparse_gated_gb300 import workloads as wl
    from oracle import bsfa_oracle as orc
    Hq, Hkv, d, Bq, Bk = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bq"], cfg["Bk"]
    g = Hq // Hkv
    nT = (cfg["cal_L"] + Bq - 1) // Bq
    rows = sorted({(h, min(i, nT - 1)) for h, i in blocks})
    acc = {r: 0.0 for r in rows}
    for n in range(cfg["n_cal"]):
        x = wl.layer_inputs(Hq, Hkv, cfg["cal_L"], d, wl.cal_seed(cfg["index"], n), device,
                            with_v=False, sink_tokens=cfg["sink_tokens"],
                            needles=cfg["cal_needles"], block=Bk)
        for h in heads:
            q64 = x.q[h].to("cpu", torch.float64).numpy()
            k64 = x.k[h // g].to("cpu", torch.float64).numpy()
            for (hh, t) in rows:
                if hh != h:
                    continue
                c = orc.candidate_maxima(q64, k64, t, Bq, Bk, 1.0 / math.sqrt(d))
                acc[(h, t)] += orc.kth_largest(c, cfg["ks"][0])
        del x
    return {(h, i): acc[(h, min(i, nT - 1))] / cfg["n_cal"] for h, i in blocks}, nT


def cpu_baseline(name, W, cnts=None):
    """The oracle on a bounded sample of the same workload on the host cores."""
    cfg, qh, kh, vh = _oracle_inputs(name, W)
    heads = sorted(qh)
    n_q = (cfg["L"] + cfg["Bq"] - 1) // cfg["Bq"]
    nT = (cfg["cal_L"] + cfg["Bq"] - 1) // cfg["Bq"]
    blocks = _sample_blocks(n_q, nT, heads, 30, 0)
    T_rows, _ = _oracle_thresholds(cfg, heads, blocks, W["q"].device)
    fl, sec, nb = oracle_sample(qh, kh, vh, heads, T_rows, blocks, cfg["Bq"], cfg["Bk"],
                                1.0 / math.sqrt(cfg["d"]))
    return {"value": round(fl / sec / 1e12, 5), "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{nb} (head, query-block) units of the 128K layer (heads {heads}, "
                      f"first/last/calibrated-boundary blocks + random), k={cfg['ks'][0]} slice, "
                      f"fp64 numpy with its BLAS on all host cores; {sec:.1f} s"}


# ----------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The fp64 oracle as it stands on the host cores: same metric and unit,
    each step a bounded sample of the workload's (head, query-block) units."""
    if rank != 0:
        return
    cfg, qh, kh, vh = _oracle_inputs(args.workload, None)
    heads = sorted(qh)
    n_q = (cfg["L"] + cfg["Bq"] - 1) // cfg["Bq"]
    nT = (cfg["cal_L"] + cfg["Bq"] - 1) // cfg["Bq"]
    steps = [_sample_blocks(n_q, nT, heads[:1], 1, 100 + s) for s in range(args.warmup + args.steps)]
    allb = sorted({b for st in steps for b in st})
    T_rows, _ = _oracle_thresholds(cfg, heads[:1], allb, "cpu")
    for st in steps[:args.warmup]:
        oracle_sample(qh, kh, vh, heads, T_rows, st[:1], cfg["Bq"], cfg["Bk"], 1 / math.sqrt(cfg["d"]))
    tot_f, tot_s, tot_b = 0.0, 0.0, 0
    for st in steps[args.warmup:]:
        f, s, b = oracle_sample(qh, kh, vh, heads, T_rows, st, cfg["Bq"], cfg["Bk"],
                                1 / math.sqrt(cfg["d"]))
        tot_f, tot_s, tot_b = tot_f + f, tot_s + s, tot_b + b
    val = tot_f / tot_s / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 5), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * tot_s / args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "sample": "per step: query blocks of head 0"},
            "cpu_baseline": {"value": round(val, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{tot_b} (head, query-block) units over {args.steps} "
                                       f"steps, fp64 numpy"},
            "e2e": {"value": round(val, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b-L131072")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--shard", default="replica", choices=["replica", "heads"],
                    help="replica: every rank runs the whole layer (weak scaling); heads: "
                         "the KV-head groups of the layer are split over the ranks (strong)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
