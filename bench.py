"""Benchmark of the fused-MoE layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one MoE-layer forward (count -> scatter + FP8 quant -> grouped FP8 GEMM w13
with SiLU-and-mul requant -> grouped FP8 GEMM w2 -> gather + top-k weight-and-reduce,
under the chunking loop) over one batch of seeded synthetic tokens already resident in
HBM. Default workload: the Qwen3-30B-A3B-shaped layer at prefill size (M=8192 tokens,
hidden 2048, moe intermediate 768, 128 experts, top-8, Zipf-skewed routing). The timed
steps cycle through --routings (default 5) routing batches drawn with consecutive router
seeds, so the number averages over which experts are hot.

Prints ONE JSON line (rank 0). With N > 1 (torchrun, one process per GPU) every rank
runs its own batch (weak scaling, no data-path collective); the time is the max over
ranks. `--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "moe_expert_layer_count_gb300", "csrc")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=mi.QWEN3_PREFILL.name, choices=sorted(mi.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step from a CUDA graph captured once per routing batch")
    ap.add_argument("--routings", type=int, default=5,
                    help="routing batches the timed steps cycle through (router seeds seed..seed+R-1)")
    return ap.parse_args()


def max_over_ranks(ms, world, device):
    """The step time of the job: the slowest rank's (all ranks get it)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s: every rank processes its own batch of tokens_per_rank
    (weak scaling), in the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, src="fallback")


# ------------------------------------------------------------------ algorithmic work
def algorithmic(li, counts_per_chunk):
    """Algorithmic bytes / flops per step (valid rows only; padding, re-reads and
    weight re-streams beyond one per chunk are not credited)."""
    wl = li.wl
    M, K, N, topk = wl.M, wl.K, wl.N, wl.topk
    R = int(sum(int(c.sum()) for c in counts_per_chunk))
    n_slots = M * topk
    a = {}
    a["count_bytes"] = n_slots * 4 + (wl.E * 4 if wl.local_experts else 0)
    # scatter: ids read (counting + ranking), x read once, FP8 rows + scales written, src2dst
    a["scatter_bytes"] = M * K * 2 + R * K + R * (K // 128) * 4 + n_slots * 4 * 2
    a["gather_bytes"] = R * K * 2 + M * K * 2 + n_slots * 8
    if N:
        a["gemm1_flops"] = 2.0 * R * (2 * N) * K
        a["gemm2_flops"] = 2.0 * R * K * N
        touched = sum(int((c > 0).sum()) for c in counts_per_chunk)
        a["weight_bytes"] = touched * (3 * N * K + (2 * N // 128) * (K // 128) * 4 + (K // 128) * (N // 128) * 4)
    a["R"] = R
    return a


def src_hash(fname):
    with open(os.path.join(CSRC, fname), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch for `kernel` on `workload` from the committed ncu summary,
    or None when absent or taken on a different version of the kernel's source."""
    path = os.path.join(PROFILES, "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[workload][kernel]
        if rec["src_sha"] != src_hash(rec["src"]):
            return None
        return float(rec["bytes_per_launch"])
    except Exception:
        return None


# -------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [r for t, r in self.rows if self.t_on and self.t_on <= t <= (self.t_off or t)]
        if not rows:
            rows = [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------------------ our arm
def run_count_only(args, world, local_rank):
    """The count step alone (count_expert_num_tokens) over 2^20 (or 2^23) tokens of top-8
    ids. 2^20 tokens of ids (33.5 MB) fit in L2, so L2 is flushed (a 256 MB write) before
    every timed step; 2^23 (268 MB) exceed it and need no flush. Each step is timed by its
    own events."""
    import torch

    import moe_expert_layer_count_gb300 as moe
    moe.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = mi.WORKLOADS[args.workload]
    ids_np, _ = mi.count_only_routing(wl)
    ids = torch.from_numpy(ids_np).to(dev)
    flush_l2 = ids_np.nbytes < (200 << 20)
    cnt = torch.empty(wl.El, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20 if flush_l2 else 1, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(i_ids=ids):
        moe.moe_count_expert_tokens(i_ids, wl.E, wl.El, None, expert_num_tokens=cnt, err_count=err)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clk = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                       if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank)
    clk.start()
    clk.mark_on()
    l0 = moe.moe_kernel_launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in evs:
        if flush_l2:
            flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clk.mark_off()
    clk.stop()
    launches = moe.moe_kernel_launch_count() - l0
    ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs) / len(evs), world, dev)
    nbytes = wl.M * wl.topk * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    pk = peaks()
    # end to end: the ids copied in from pinned memory, the counts read back, every step
    ih = torch.from_numpy(ids_np).pin_memory()
    ch = torch.empty(wl.El, dtype=torch.int32).pin_memory()
    for _ in range(3):
        ids.copy_(ih, non_blocking=True)
        step()
        ch.copy_(cnt, non_blocking=True)
    torch.cuda.synchronize()
    n_e2e = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        ids.copy_(ih, non_blocking=True)
        step()
        ch.copy_(cnt, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / n_e2e
    return {
        "metric": "MoE-layer tokens/s", "value": round(job_throughput(wl.M, world, ms), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic: seeded N(0,1) router logits, top-8 of 128 experts",
        "config": workload_config(wl, world),
        "gpu_launches": int(launches), "clocks": clk.summary(),
        "roofline": {"kernel": "count", "bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"],
                     "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                     "peak_source": "measured copy bandwidth" if pk["src"] == "measured" else "fallback",
                     "traffic": None, "algorithmic_per_launch": float(nbytes)},
        "kernels": {"count": {"us_per_step": round(ms * 1e3, 2), "launches_per_step": launches / args.steps,
                              "GB/s": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm"], 4)}},
        "e2e": {"value": round(job_throughput(wl.M, world, ms_e2e), 1), "unit": "tokens/s",
                "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": int(ih.numel() * 4),
                "d2h_bytes_per_step": int(ch.numel() * 4), "steps": n_e2e},
    }


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import moe_expert_layer_count_gb300 as moe
    moe.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = mi.WORKLOADS[args.workload]
    li = mi.make_layer_inputs(wl)
    E, El, M, K, N, topk = wl.E, wl.El, wl.M, wl.K, wl.N, wl.topk
    chunk = wl.chunk

    def D(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    # routing variation: timed step i runs routing batch i % R (router seeds seed .. seed+R-1,
    # the same tokens and weights); batch 0 is the workload's own routing
    R = max(1, args.routings)
    host_routes = [(li.topk_ids, li.topk_weights)] + [mi.route(M, E, topk, wl.seed + b, wl.zipf_s)
                                                      for b in range(1, R)]
    routes = [(D(i_), D(w_)) for i_, w_ in host_routes]
    x = D(li.x)
    ids, tw = routes[0]
    emap = None if li.expert_map is None else D(li.expert_map)
    permute_only = N == 0
    stream = torch.cuda.current_stream()
    cmax = min(chunk, M)
    out = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    if not permute_only:
        w13, s13, w2, s2 = D(li.w13), D(li.w13_scale), D(li.w2), D(li.w2_scale)
        ws = torch.empty(moe.moe_workspace_size(cmax, K, N, topk, El), dtype=torch.uint8, device=dev)

        def step(i=0):
            ids_i, tw_i = routes[i % R]
            moe.moe_forward_chunked(x, ids_i, tw_i, w13, s13, w2, s2, E, expert_map=emap, chunk_size=chunk,
                                    out=out, workspace=ws)
    else:
        cap = moe.moe_rp_cap(M, topk, El)
        A = torch.empty(cap, K, dtype=torch.uint8, device=dev)
        SA = torch.empty(cap, K // 128, dtype=torch.float32, device=dev)
        offs = torch.empty(El + 1, dtype=torch.int32, device=dev)
        s2d = torch.empty(M, topk, dtype=torch.int32, device=dev)
        cnt = torch.empty(El, dtype=torch.int32, device=dev)
        sws = torch.empty(moe.moe_scatter_workspace_size(M, topk, El), dtype=torch.uint8, device=dev)
        # identity experts: Y is the bf16 permuted copy of x, one per routing batch
        Ys = [moe.moe_scatter(x, i_, w_, E, El, moe.moe_count_expert_tokens(i_, E, El, emap), emap,
                              quant=moe.MOE_QUANT_NONE)[0] for i_, w_ in routes]
        Y = Ys[0]

        def step(i=0):
            ids_i, tw_i = routes[i % R]
            moe.moe_scatter(x, ids_i, tw_i, E, El, cnt, emap, rp_cap=cap, a_out=A, a_scale=SA, expert_offsets=offs,
                            src2dst=s2d, workspace=sws, count_here=True)
            moe.moe_gather_weight_reduce(Ys[i % R], s2d, tw_i, out=out)

    # per-chunk counts (host side, for the algorithmic work only)
    counts = []
    for c0 in range(0, M, chunk):
        c = torch.zeros(El, dtype=torch.int32, device=dev)
        moe.moe_count_expert_tokens(ids[c0:c0 + chunk].contiguous(), E, El, emap, expert_num_tokens=c)
        counts.append(c.cpu().numpy())
    work = algorithmic(li, counts)

    clk = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                       if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank)
    run = step
    graph_launches = None
    if args.graph:
        # one CUDA graph per routing batch, captured on the same static buffers the eager
        # steps use; a replay launches the step's kernels without the host API in between
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for i in range(R):
                step(i)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        lc0 = moe.moe_kernel_launch_count()
        graphs = []
        for b in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(b)
            graphs.append(g)
        graph_launches = (moe.moe_kernel_launch_count() - lc0) // R  # kernels in one step's graph
        run = lambda i: graphs[i % R].replay()
    clk.start()
    for i in range(args.warmup):
        run(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = moe.moe_kernel_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk.mark_on()
    e0.record(stream)
    for i in range(args.steps):
        run(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk.mark_off()
    launches = (moe.moe_kernel_launch_count() - l0) if graph_launches is None else graph_launches * args.steps
    ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ms, world, dev)
    clk.stop()

    # ---- per-kernel breakdown on the same stream (separate loop, same calls) ----
    kern = kernel_breakdown(moe, torch, stream, li, x, ids, tw, emap, dev, args, permute_only,
                            locals().get("w13"), locals().get("s13"), locals().get("w2"), locals().get("s2"))

    # ---- end to end: pinned host inputs -> device -> layer -> host output, per step ----
    e2e = None
    if not args.no_e2e:
        layer = None if permute_only else dict(w13=w13, s13=s13, w2=w2, s2=s2, emap=emap, chunk=chunk)
        e2e = end_to_end(moe, torch, stream, li, dev, args, step, x, routes, out, layer, host_routes)

    value = job_throughput(M, world, ms)
    pk = peaks()
    roof = roofline(kern, work, pk, wl)
    line = {
        "metric": "MoE-layer tokens/s",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if not permute_only else "bf16/fp8_e4m3",
        "data": "synthetic: seeded N(0,1) bf16 tokens, N(0,1)+Zipf router logits, random-init N(0,0.02) "
                "weights quantised to FP8 e4m3 with 128x128 block scales",
        "config": workload_config(wl, world),
        "run": {"cuda_graph": bool(args.graph),
                "routing_batches": f"{R} (router seeds {wl.seed}..{wl.seed + R - 1}, step i runs batch i % {R}; "
                                   f"per-kernel breakdown and roofline on batch 0)",
                "touched_weight_mb": round(work.get("weight_bytes", 0) / 1e6, 1)},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "roofline": roof,
        "kernels": kern["table"],
        "scatter_gbs": kern["table"].get("scatter", {}).get("GB/s"),
        "gather_gbs": kern["table"].get("gather", {}).get("GB/s"),
        "gemm_tflops": kern["table"].get("gemm1", {}).get("TFLOP/s"),
        "e2e": e2e,
    }
    return line


def kernel_breakdown(moe, torch, stream, li, x, ids, tw, emap, dev, args, permute_only, w13, s13, w2, s2):
    """Time each stage of one chunk-loop pass with CUDA events on the launching stream,
    calling the same entry points the layer's chunk loop calls."""
    wl = li.wl
    E, El, M, K, N, topk, chunk = wl.E, wl.El, wl.M, wl.K, wl.N, wl.topk, wl.chunk
    cmax = min(chunk, M)
    cap = moe.moe_rp_cap(cmax, topk, El)
    cnt = torch.empty(El, dtype=torch.int32, device=dev)
    A = torch.empty(cap, K, dtype=torch.uint8, device=dev)
    SA = torch.empty(cap, K // 128, dtype=torch.float32, device=dev)
    offs = torch.empty(El + 1, dtype=torch.int32, device=dev)
    s2d = torch.empty(cmax, topk, dtype=torch.int32, device=dev)
    sws = torch.empty(moe.moe_scatter_workspace_size(cmax, topk, El), dtype=torch.uint8, device=dev)
    Y = torch.empty(cap, K, dtype=torch.bfloat16, device=dev)
    out = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    if not permute_only:
        H = torch.empty(cap, N, dtype=torch.uint8, device=dev)
        HS = torch.empty(cap, N // 128, dtype=torch.float32, device=dev)
        fused = FUSED_SILU
        C1 = None if fused else torch.empty(cap, 2 * N, dtype=torch.float32, device=dev)
    stages = ["scatter"] + ([] if permute_only else (["gemm1"] + ([] if FUSED_SILU else ["silu"]) +
                                                      ["gemm2"])) + ["gather"]
    reps = max(3, min(args.steps, 20))
    times = {s: 0.0 for s in stages}
    launches = {s: 0 for s in stages}
    ev = lambda: torch.cuda.Event(enable_timing=True)
    n_chunks = (M + chunk - 1) // chunk
    for it in range(reps + 2):
        # a bounded device-side sleep gives the host a head start, so that the events
        # below measure back-to-back kernels, not host enqueue gaps
        torch.cuda._sleep(int(2e9 * max(1e-3, 60e-6 * len(stages) * n_chunks)))
        recs = []
        for c0 in range(0, M, chunk):
            Mc = min(chunk, M - c0)
            capc = moe.moe_rp_cap(Mc, topk, El)
            e = [ev() for _ in range(len(stages) + 1)]
            xi, ii, wi = x[c0:c0 + Mc], ids[c0:c0 + Mc], tw[c0:c0 + Mc]
            n0 = moe.moe_kernel_launch_count()
            marks = []
            e[0].record(stream)
            # the count step runs inside the scatter's histogram pass, as in the chunk loop
            moe.moe_scatter(xi, ii, wi, E, El, cnt, emap, rp_cap=capc, a_out=A[:capc], a_scale=SA[:capc],
                            expert_offsets=offs, src2dst=s2d[:Mc], workspace=sws, count_here=True)
            marks.append(moe.moe_kernel_launch_count())
            e[1].record(stream)
            j = 1
            if permute_only:
                Yv = Y[:capc]
            else:
                if FUSED_SILU:
                    moe.moe_grouped_gemm_fp8(A[:capc], SA[:capc], w13, s13, offs, moe.MOE_EPI_SILU_MUL_QUANT,
                                             out=H[:capc], out_scale=HS[:capc])
                else:
                    moe.moe_grouped_gemm_fp8(A[:capc], SA[:capc], w13, s13, offs, moe.MOE_EPI_F32, out=C1[:capc])
                    marks.append(moe.moe_kernel_launch_count())
                    j += 1
                    e[j].record(stream)
                    moe.moe_silu_mul_quant(C1[:capc], offs, h=H[:capc], h_scale=HS[:capc])
                marks.append(moe.moe_kernel_launch_count())
                j += 1
                e[j].record(stream)
                moe.moe_grouped_gemm_fp8(H[:capc], HS[:capc], w2, s2, offs, moe.MOE_EPI_BF16, out=Y[:capc])
                marks.append(moe.moe_kernel_launch_count())
                j += 1
                e[j].record(stream)
                Yv = Y[:capc]
            moe.moe_gather_weight_reduce(Yv, s2d[:Mc], wi, out=out[c0:c0 + Mc])
            marks.append(moe.moe_kernel_launch_count())
            j += 1
            e[j].record(stream)
            recs.append((e, n0, marks))
        torch.cuda.synchronize()
        if it >= 2:
            for e, n0, marks in recs:
                prev = n0
                for si, s in enumerate(stages):
                    times[s] += e[si].elapsed_time(e[si + 1])
                    launches[s] += marks[si] - prev
                    prev = marks[si]
    table = {}
    for s in stages:
        us = times[s] / reps * 1e3
        table[s] = {"us_per_step": round(us, 2), "launches_per_step": launches[s] // reps}
    return {"table": table}


def roofline(kern, work, pk, wl):
    t = kern["table"]
    for s, key in (("scatter", "scatter_bytes"), ("gather", "gather_bytes")):
        if s in t and t[s]["us_per_step"] > 0:
            t[s]["GB/s"] = round(work[key] / (t[s]["us_per_step"] * 1e-6) / 1e9, 1)
            t[s]["hbm_frac"] = round(t[s]["GB/s"] / pk["hbm"], 4)
    fp8_peak = 2.0 * pk["bf16"]   # dense FP8 = 2x dense bf16 (nominal ratio 4.5 / 2.25 PFLOP/s)
    for s, key in (("gemm1", "gemm1_flops"), ("gemm2", "gemm2_flops")):
        if s in t and t[s]["us_per_step"] > 0:
            t[s]["TFLOP/s"] = round(work[key] / (t[s]["us_per_step"] * 1e-6) / 1e12, 1)
            t[s]["tensor_frac"] = round(t[s]["TFLOP/s"] / fp8_peak, 4)
    dom = max(t, key=lambda s: t[s]["us_per_step"])
    launches = max(1, t[dom]["launches_per_step"])
    if dom.startswith("gemm"):
        achieved = t[dom]["TFLOP/s"]
        traffic = recorded_traffic(dom, wl.name)
        return {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                "peak_source": f"{pk['src']} bf16 {pk['bf16']} TFLOP/s x 2 (dense fp8/bf16 nominal ratio)",
                "traffic": None if traffic is None else traffic,
                "algorithmic_per_launch": work[dom + "_flops"] / launches}
    achieved = t[dom].get("GB/s")
    traffic = recorded_traffic(dom, wl.name)
    return {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm"], 4) if achieved else None,
            "peak_source": f"{pk['src']} copy bandwidth", "traffic": traffic,
            "algorithmic_per_launch": work[dom + "_bytes"] / launches}


FUSED_SILU = True  # GEMM1 applies SiLU-and-mul + FP8 requant in its epilogue (as the chunk loop does)


def end_to_end(moe, torch, stream, li, dev, args, step_dev, x, routes, out, layer, host_routes):
    """Same metric through the public API with host buffers: every step copies that
    step's inputs from pinned host memory to the device and the output back.

    The layer workloads call moe_forward_host, the C-ABI entry point that takes host
    buffers: successive steps are issued back to back, as a serving loop issues batches,
    so a step's copies run on the library's copy streams while its neighbours compute.
    The timed region starts on an idle device and ends once the last output copy has
    completed. The permute-only workload (no layer entry point) copies around its two
    calls on the compute stream."""
    wl = li.wl
    xh = torch.from_numpy(np.ascontiguousarray(li.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    ihs = [torch.from_numpy(np.ascontiguousarray(i_)).pin_memory() for i_, _ in host_routes]
    whs = [torch.from_numpy(np.ascontiguousarray(w_)).pin_memory() for _, w_ in host_routes]
    ih, wh = ihs[0], whs[0]
    R = len(host_routes)
    oh = [torch.empty(wl.M, wl.K, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    if layer is not None:
        El, N2, _ = layer["w13"].shape
        hws = torch.empty(moe.moe_host_workspace_size(wl.M, wl.K, N2 // 2, wl.topk, El, layer["chunk"]),
                          dtype=torch.uint8, device=dev)

        def step(i):
            moe.moe_forward_host(xh, ihs[i % R], whs[i % R], layer["w13"], layer["s13"], layer["w2"], layer["s2"],
                                 wl.E,
                                 expert_map=layer["emap"], chunk_size=layer["chunk"], out=oh[i & 1],
                                 workspace=hws, stream=stream)

        def drain():
            moe.moe_host_wait(stream)
    else:
        def step(i):
            ids_i, tw_i = routes[i % R]
            x.copy_(xh, non_blocking=True)
            ids_i.copy_(ihs[i % R], non_blocking=True)
            tw_i.copy_(whs[i % R], non_blocking=True)
            step_dev(i)
            oh[i & 1].copy_(out, non_blocking=True)

        def drain():
            pass

    for i in range(max(3, args.warmup)):
        step(i)
    drain()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    drain()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(wl.M / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(xh.numel() * 2 + ih.numel() * 4 + wh.numel() * 4),
            "d2h_bytes_per_step": int(oh[0].numel() * 2), "steps": steps,
            "api": "moe_forward_host (pipelined)" if layer is not None else "moe_scatter + moe_gather_weight_reduce"}


# ------------------------------------------------------------------ config
def workload_config(wl, world):
    """The JSON line's `config`: the workload, its shape and the L2 rule, the same for
    both arms."""
    c = {"workload": wl.name, "M": wl.M, "hidden": wl.K}
    if wl.N:
        c["moe_intermediate"] = wl.N
    c.update({"experts": wl.E, "local_experts": wl.El, "topk": wl.topk, "chunk_size": wl.chunk,
              "routing": f"zipf s={wl.zipf_s}" if wl.zipf_s else "uniform",
              "parallelism": f"replicas x{world} (one independent batch per GPU)"})
    if mi.is_count_only(wl):
        c["step"] = "count only"
        c["l2"] = ("flushed before every timed step (256 MB write); each step timed by its own events"
                   if wl.M * wl.topk * 4 < (200 << 20) else
                   "inputs larger than L2 (268 MB of ids, the 2^20-token routing repeated 8 times); no flush")
    elif wl.N:
        c["l2"] = "inputs larger than L2: the touched experts' FP8 weights alone exceed the 129 MB L2"
    else:
        c["l2"] = "inputs larger than L2: hidden states + permuted rows + unpermuted output exceed it"
    return c


# ------------------------------------------------------------------- CPU oracle
ORACLE_BUDGET_S = 90.0  # wall time the reference arm's timed + warm-up oracle calls may take


def _oracle_inputs(wl):
    count_only = mi.is_count_only(wl)
    if count_only:  # only the routing is needed
        ids, w = mi.count_only_routing(wl)
        return mi.LayerInputs(wl, np.zeros((wl.M, 0), np.uint16), ids, w, None)
    return mi.make_layer_inputs(wl)


def _oracle_call(wl, li, m, parallel):
    """One oracle pass over the first m tokens of the workload (the OpenMP build when
    parallel; only the layer has a multi-threaded row loop)."""
    import oracle
    if mi.is_count_only(wl):
        oracle.count(li.topk_ids[:m], wl.E, wl.El)
    elif wl.N:
        oracle.forward_chunked(li.x[:m], li.topk_ids[:m], li.topk_weights[:m], li.w13, li.w13_scale, li.w2,
                               li.w2_scale, wl.E, expert_map=li.expert_map, chunk_size=wl.chunk, parallel=parallel)
    else:
        r = oracle.scatter(li.x[:m], li.topk_ids[:m], li.topk_weights[:m], wl.E, wl.El, li.expert_map)
        oracle.gather(mi.bf16_bits(np.zeros((r["a"].shape[0], wl.K), np.float32)), r["src2dst"],
                      li.topk_weights[:m])


def oracle_sample(wl, calls, budget_s=ORACLE_BUDGET_S):
    """The token sample both CPU legs time: the first m tokens, m the largest power of two
    (at most M) whose OpenMP oracle pass, repeated `calls` times, fits in budget_s
    (estimated from a calibration pass). Returns (inputs, m)."""
    li = _oracle_inputs(wl)
    m0 = min(wl.M, 8 if wl.N else 1024)
    t0 = time.perf_counter()
    _oracle_call(wl, li, m0, True)
    per_token = max(1e-9, (time.perf_counter() - t0) / m0)
    fit = budget_s / max(1, calls) / per_token
    m = 1
    while m * 2 <= min(wl.M, fit):
        m *= 2
    return li, max(1, min(m, wl.M))


def _timed(wl, li, m, parallel, min_s):
    """Tokens/s of repeated oracle passes over m tokens, at least one pass and min_s."""
    n, t = 0, 0.0
    while n == 0 or t < min_s:
        t0 = time.perf_counter()
        _oracle_call(wl, li, m, parallel)
        t += time.perf_counter() - t0
        n += 1
    return m * n / t, n, t


def cpu_baseline(wl, calls):
    """The oracle as it stands on the host cores: its OpenMP build over all cores (the
    reported value) and the single-threaded checker, on the reference arm's sample."""
    import oracle
    li, m = oracle_sample(wl, calls)
    par = bool(wl.N) and not mi.is_count_only(wl)
    v, n, t = _timed(wl, li, m, par, 8.0)
    v1, n1, t1 = _timed(wl, li, m, False, 8.0)
    cores = oracle.num_threads(True) if par else 1
    return {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {m} of {wl.M} tokens of {wl.name}, {n} passes in {t:.1f} s "
                      f"({'OpenMP C oracle' if par else 'single-threaded C oracle'})",
            "single_thread": {"value": round(v1, 3), "unit": "tokens/s", "cores": 1,
                              "sample": f"first {m} tokens, {n1} passes in {t1:.1f} s"}}


def run_reference(args):
    """The reference arm: the CPU oracle (OpenMP build, all host cores) on the same token
    sample the CPU-baseline leg times, W warm-up and K timed passes."""
    import oracle
    wl = mi.WORKLOADS[args.workload]
    li, m = oracle_sample(wl, args.warmup + args.steps)
    par = bool(wl.N) and not mi.is_count_only(wl)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _oracle_call(wl, li, m, par)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    s = sum(times)
    value = m * len(times) / s
    cores = oracle.num_threads(True) if par else 1
    return {"impl": "reference", "metric": "MoE-layer tokens/s", "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(s / len(times) * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp64 (oracle)", "data": "synthetic",
            "config": workload_config(wl, args.gpus),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {m} of {wl.M} tokens per pass "
                                       f"({'OpenMP C oracle' if par else 'single-threaded C oracle'})"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if mi.is_count_only(mi.WORKLOADS[args.workload]):
        line = run_count_only(args, world, local_rank)
    else:
        line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(mi.WORKLOADS[args.workload], args.warmup + args.steps)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
