"""Benchmark of the DFlash 2 selection + verify path on GB300.

One step = one pass of the whole hot path over one batch: dflash2_topk16 ->
dflash2_ctx_gate -> dflash2_pair_score_walk -> dflash2_verify on B requests
of K drafted positions each.  The metric is draft blocks per second (one block
= one request's K-position block taken through the four calls), measured on
seeded synthetic inputs that are resident in HBM; 3 input sets rotate and
each is larger than L2, so every step streams its logits from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 27b_greedy] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the
workload (the path has no cross-request exchange); value = blocks of all
ranks / max-over-ranks time.  `--impl reference` times the CPU oracle on the
host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft blocks/sec (topk+select+verify) at B=64,V=151936; % of HBM roofline"
UNIT = "blocks/s"
KERNEL_SOURCES = {  # every file of the library each kernel is compiled from
    "k_topk16": ["common.cuh", "host.hpp", "rowscan.cuh", "filter.cuh", "wide.cuh", "topk16.cu"],
    "k_verify": ["common.cuh", "host.hpp", "rowscan.cuh", "filter.cuh", "wide.cuh", "verify.cu"],
    "k_gate_tc": ["common.cuh", "host.hpp", "tc.cuh", "gate.cu"],
    "k_pair_score_walk": ["common.cuh", "host.hpp", "walk.cu"],
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default="27b_greedy")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-kernel-pass", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of graph replays")
    ap.add_argument("--graph-steps", type=int, default=6,
                    help="consecutive steps captured in one CUDA graph (a multiple of the 3 input sets)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _code_only(text):
    """C++ source without comments, trailing blanks and empty lines (edits to comments keep the hash)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def max_over_ranks(x, dev, world):
    """The largest of every rank's x (the job ends when its slowest replica does)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(B, world, steps, seconds):
    """Draft blocks per second of the whole job: every replica runs B requests per step."""
    return B * world * steps / seconds


def kernel_source_sha(kernel):
    h = hashlib.sha256()
    for n in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "dflash_draft_selection_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_t or m_sha.group(1) != kernel_source_sha(kernel):
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(prefix="clocks", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for r in csv.reader(f):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------- workload ----
def algorithmic_bytes(shp):
    """Bytes the method must move per launch of each kernel (inputs it reads + outputs it writes)."""
    e = 2 if "bfloat16" in str(shp.dtype) else 4
    B, K, V, Hd, D = shp.B, shp.K, shp.V, shp.hidden, shp.D
    nc = 16
    return {
        "k_topk16": B * K * V * e + B * K * (nc * 8 + 4),
        "k_verify": B * (K + 1) * V * e + B * (K * (nc * 8 + 8) + (K + 1) * 8),
        "k_gate_tc": (B * K * Hd + D * Hd) * e + B * K * D * 4,
        "k_pair_score_walk": B * (1 + nc * (K - 1) + nc * K) * D * e + B * K * (D * 4 + nc * nc * 4 + nc * 8),
    }


class Chain:
    """Inputs, outputs and workspaces of one step; step() makes the four calls."""

    def __init__(self, shp, dev, nsets=3):
        import torch

        import dflash_draft_selection_gb300 as d2
        from dflash_draft_selection_gb300 import synth
        self.d2, self.torch, self.shp, self.dev = d2, torch, shp, dev
        B, K = shp.B, shp.K
        self.sets = []
        for i in range(nsets):
            s = synth.Shape(**{**shp.__dict__, "seed": shp.seed + 1000 * i})
            self.sets.append(synth.make_inputs(s, device=dev, with_conv=False))
        base = self.sets[0]
        self.A, self.Bt, self.Wg = base.A, base.Bt, base.Wg          # model weights: shared by all sets
        self.sampled = shp.temperature > 0
        p = base.params
        self.params = d2.sampling_params(p["temperature"], p["top_k"], p["top_p"], device=dev) if self.sampled else None
        e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device=dev)
        self.cand, self.U, self.lse = e(B * K, 16, dt=torch.int32), e(B * K, 16), e(B * K)
        self.gate = e(B * K, shp.D)
        self.pt, self.ps = e(B, K, dt=torch.int32), e(B, K, dt=torch.int32)
        self.q, self.S = e(B, K, 16), e(B, K, 16, 16)
        self.acc, self.out, self.st = e(B, dt=torch.int32), e(B, K + 1, dt=torch.int32), e(B, dt=torch.int32)
        self.ws_topk = d2.Workspace.for_topk16(B * K, dev)
        self.ws_verify = d2.Workspace.for_verify(B, K, dev)

    def call(self, which, inp):
        d2, B, K = self.d2, self.shp.B, self.shp.K
        pg = self.params
        if which == "k_topk16":
            d2.topk16(inp.draft_logits, params=pg, rows_per_param=K, ws=self.ws_topk,
                      out=(self.cand, self.U, self.lse))
        elif which == "k_gate_tc":
            d2.ctx_gate(inp.h, self.Wg, out=self.gate)
        elif which == "k_pair_score_walk":
            d2.pair_score_walk(self.cand.view(B, K, 16), self.U.view(B, K, 16), inp.last_tok, self.A, self.Bt,
                               self.gate.view(B, K, -1), params=pg, u_walk=inp.u_walk if self.sampled else None,
                               out=(self.pt, self.ps, self.q, self.S))
        else:
            d2.verify(inp.target_logits, self.pt, self.cand.view(B, K, 16), self.q, self.ps, params=pg,
                      u_acc=inp.u_acc if self.sampled else None, u_res=inp.u_res if self.sampled else None,
                      ws=self.ws_verify, out=(self.acc, self.out, self.st))

    ORDER = ("k_topk16", "k_gate_tc", "k_pair_score_walk", "k_verify")

    def run(self, inp):
        """One pass of the path on one stream.  The library launches ctx_gate so that it may run in
        topk16's tail (it needs only the drafter's hidden state; programmatic dependent launch)."""
        for k in self.ORDER:
            self.call(k, inp)

    def step(self, i):
        self.run(self.sets[i % len(self.sets)])


def run_ours(args, rank, world, local):
    import torch

    from dflash_draft_selection_gb300 import synth
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        dist.barrier()
    shp = synth.WORKLOADS[args.config]
    chain = Chain(shp, dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(max(args.warmup, 3)):
        chain.step(i)
    torch.cuda.synchronize()

    # One graph of S consecutive steps (step i reads input set i mod 3), so that programmatic
    # dependent launches also link one step's verify to the next step's topk16; single-step
    # graphs cover K mod S.
    graphs, multi = [], None
    nsets = len(chain.sets)
    S = 1 if args.graph_steps <= 1 else max(nsets, args.graph_steps // nsets * nsets)
    if not args.eager:
        cap = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(cap):
            for i in range(nsets):
                chain.step(i)          # warm the capture stream
            cap.synchronize()
            for i in range(nsets):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    chain.step(i)
                graphs.append(g)
            if S > 1:
                multi = torch.cuda.CUDAGraph()
                with torch.cuda.graph(multi, stream=cap):
                    for i in range(S):
                        chain.step(i)
        for g in graphs:
            g.replay()
        if multi is not None:
            multi.replay()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps ----
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if graphs:
        full = args.steps // S if multi is not None else 0
        for _ in range(full):
            multi.replay()
        for i in range(full * S, args.steps):
            graphs[i % nsets].replay()
    else:
        for i in range(args.steps):
            chain.step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), dev, world)
    ms_per_step = ms / args.steps
    value = whole_job_rate(shp.B, world, args.steps, ms / 1e3)

    # ---- per-kernel durations: eager steps queued behind a sleep kernel ----
    kern = {} if args.no_kernel_pass else kernel_pass(chain, stream, min(args.steps, 400))
    algo = algorithmic_bytes(shp)
    peak, peak_kind = measured_peaks()
    roof = None
    if kern:
        roof = roofline(kern, algo, ms_per_step, peak, peak_kind, args.config)

    # ---- the other workloads (sampled; stress) and the drafter-side conv, each with its own roofline ----
    aux = None
    if not args.no_kernel_pass:
        aux = {"conv2tap": time_conv(dev, peak), "dynconv2tap": time_dynconv(dev, peak)}
        for name in AUX_WORKLOADS:
            if name != args.config:
                aux[name] = time_workload(name, dev, peak, peak_kind)
        aux["lmhead_topk16"] = time_lmhead(dev)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(chain, shp, dev, stream, min(args.steps, 200), world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(shp, budget_s=10.0)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if "bfloat16" in str(shp.dtype) else "f32",
                "data": "synthetic (seeded; Gumbel+spike logits, 85% top-1 mass; random-init tables)",
                "config": {"workload": args.config, "B": shp.B, "K": shp.K, "V": shp.V, "hidden": shp.hidden,
                           "D": shp.D, "sampling": "greedy" if shp.temperature == 0 else
                           f"T={shp.temperature},top_k={shp.top_k},top_p={shp.top_p}",
                           "l2": "inputs larger than L2 (292 MB of logits per step), 3 rotating input sets",
                           "timing": (f"CUDA graphs of {S} consecutive steps of the 4-call chain (programmatic "
                                      "dependent launches: ctx_gate runs in topk16's tail, each kernel is "
                                      "scheduled before its predecessor completes)") if graphs else "eager launches",
                           "parallelism": f"replicas x{world}"},
                "gpu_launches": 4 * args.steps, "clocks": clk, "roofline": roof, "e2e": e2e, "cpu_baseline": cpu,
                "aux": aux}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


AUX_WORKLOADS = ("27b_greedy", "27b_sampled", "27b_nucleus", "stress")


def kernel_pass(chain, stream, n):
    """Mean duration of each kernel of the step over n eager steps, queued behind a sleep kernel so that
    the CPU enqueues ahead of the GPU; CUDA events on the launching stream between the calls."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(Chain.ORDER) + 1)] for _ in range(n)]
    torch.cuda._sleep(int(1e6 * n))
    for i in range(n):
        inp = chain.sets[i % len(chain.sets)]
        evs[i][0].record(stream)
        for j, k in enumerate(Chain.ORDER):
            chain.call(k, inp)
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize()
    return {k: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n)) / n for j, k in enumerate(Chain.ORDER)}


def roofline(kern, algo, ms_per_step, peak, peak_kind, workload):
    """The dominant scan's HBM roofline (algorithmic bytes / its mean launch time) and the whole step's."""
    dom = max(("k_topk16", "k_verify"), key=lambda k: kern[k])
    achieved = algo[dom] / (kern[dom] * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(dom, workload), "peak_source": peak_kind,
            "algorithmic_bytes": algo[dom], "avg_launch_us": round(kern[dom] * 1e3, 2),
            "kernels_us": {k: round(v * 1e3, 2) for k, v in kern.items()},
            "step_bytes_frac_of_peak": round(sum(algo.values()) / (ms_per_step * 1e-3) / 1e9 / peak, 4)}


def time_workload(name, dev, peak, peak_kind, steps=30):
    """Another workload's step: graphs of 3 consecutive steps (3 rotating input sets, every set larger
    than L2) timed with CUDA events, then the per-kernel pass."""
    import torch

    from dflash_draft_selection_gb300 import synth
    shp = synth.WORKLOADS[name]
    chain = Chain(shp, dev)
    nsets = len(chain.sets)
    cap = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(cap):
        for i in range(max(3, nsets)):
            chain.step(i)
        cap.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(nsets):
                chain.step(i)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // nsets)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_per_step = e0.elapsed_time(e1) / (reps * nsets)
    kern = kernel_pass(chain, stream, min(steps, 60))
    algo = algorithmic_bytes(shp)
    out = {"workload": name, "B": shp.B, "K": shp.K, "V": shp.V,
           "sampling": "greedy" if shp.temperature == 0 else
           f"T={shp.temperature},top_k={shp.top_k},top_p={shp.top_p}",
           "value": round(shp.B / (ms_per_step * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms_per_step, 5),
           "steps": reps * nsets, "roofline": roofline(kern, algo, ms_per_step, peak, peak_kind, name)}
    del chain, g
    torch.cuda.empty_cache()
    return out


def time_lmhead(dev, reps=10):
    """dflash2_lmhead_topk16 (the drafter's LM head fused with the top-16) at the 27B drafter's shape
    (hidden 5120, V 151936) for 448 rows (B=64, K=7) and 3840 rows (B=256, K=15): mean of `reps`
    launches with CUDA events (W is 1.56 GB, larger than L2); algorithmic FLOPs 2 * rows * hidden * V
    against the measured bf16 tensor peak (burst: the kernel is timed alone)."""
    import torch

    import dflash_draft_selection_gb300 as d2
    peaks = {}
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        peaks = json.load(open(p))
    peak = float(peaks.get("bf16_tflops", 1900.0))
    out = {"unit": "TFLOP/s", "peak": peak, "bound": "tensor", "peak_source": "measured" if peaks else "fallback"}
    g = torch.Generator(device=dev).manual_seed(11)
    hidden, V = 5120, 151936
    W = (torch.randn(V, hidden, generator=g, device=dev) / hidden ** 0.5).bfloat16()
    for rows in (448, 3840):
        h = torch.randn(rows, hidden, generator=g, device=dev).bfloat16()
        ws = d2.Workspace.for_lmhead(rows, V, dev)
        res = (torch.empty(rows, 16, dtype=torch.int32, device=dev), torch.empty(rows, 16, device=dev),
               torch.empty(rows, device=dev))
        for _ in range(3):
            d2.lmhead_topk16(h, W, ws=ws, out=res)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            d2.lmhead_topk16(h, W, ws=ws, out=res)
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / reps * 1e3
        tf = 2.0 * rows * hidden * V / (us * 1e-6) / 1e12
        out[f"rows_{rows}"] = {"avg_launch_us": round(us, 1), "achieved": round(tf, 1), "frac": round(tf / peak, 4)}
        del h, ws
    del W
    torch.cuda.empty_cache()
    return out


def time_conv(dev, peak, reps=50):
    """dflash2_conv2tap at the stress workload's conv shape ([256, 16, 5120] bf16, per-request x_prev):
    mean of `reps` launches with CUDA events; every launch streams 170 MB (more than L2)."""
    import torch

    import dflash_draft_selection_gb300 as d2
    from dflash_draft_selection_gb300 import synth
    shp = synth.WORKLOADS["stress"]
    g = torch.Generator(device=dev).manual_seed(shp.seed)
    c = synth.make_conv(shp.B, shp.K + 1, shp.hidden, shp.dtype, g, dev)
    y = torch.empty_like(c["x"])
    for _ in range(3):
        d2.conv2tap(c["x"], c["k0"], c["k1"], c["x_prev"], out=y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        d2.conv2tap(c["x"], c["k0"], c["k1"], c["x_prev"], out=y)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    n = c["x"].numel()
    algo = 4 * n * 2 + c["x_prev"].numel() * 2   # x, k0, k1 in; y out; x_prev
    gbs = algo / (us * 1e-6) / 1e9
    return {"workload": "stress conv [256, 16, 5120] bf16", "avg_launch_us": round(us, 2),
            "algorithmic_bytes": algo, "achieved": round(gbs, 1), "unit": "GB/s", "peak": peak,
            "frac": round(gbs / peak, 4), "bound": "hbm"}


def time_dynconv(dev, peak, reps=50):
    """dflash2_dynconv2tap at the stress workload's conv shape ([256, 16, 5120] bf16, group size 80:
    64 groups): the taps' projection on the tensor cores, then the conv; mean of `reps` calls with
    CUDA events.  Algorithmic bytes: x and x_prev read once, Wd, the taps and y written."""
    import torch

    import dflash_draft_selection_gb300 as d2
    from dflash_draft_selection_gb300 import synth
    shp = synth.WORKLOADS["stress"]
    B, T, H, gs = shp.B, shp.K + 1, shp.hidden, 80
    g = torch.Generator(device=dev).manual_seed(shp.seed + 1)
    x = torch.randn(B, T, H, generator=g, device=dev).to(shp.dtype)
    xp = torch.randn(B, H, generator=g, device=dev).to(shp.dtype)
    W = (torch.randn(H // gs, H, generator=g, device=dev) * (2.0 / H ** 0.5)).to(shp.dtype)
    out = (torch.empty(B, T, H // gs, dtype=torch.float32, device=dev), torch.empty_like(x))
    for _ in range(3):
        d2.dynconv2tap(x, xp, W, gs, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        d2.dynconv2tap(x, xp, W, gs, out=out)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    algo = (2 * x.numel() + xp.numel() + W.numel()) * 2 + out[0].numel() * 4
    gbs = algo / (us * 1e-6) / 1e9
    return {"workload": f"stress dynamic conv [{B}, {T}, {H}] bf16, group size {gs}", "avg_launch_us": round(us, 2),
            "algorithmic_bytes": algo, "achieved": round(gbs, 1), "unit": "GB/s", "peak": peak,
            "frac": round(gbs / peak, 4), "bound": "hbm", "launches_per_call": 2}


def run_e2e(chain, shp, dev, stream, steps, world):
    """Host-resident inputs through the public calls: every step copies its inputs from pinned host
    memory (cudaMemcpyAsync on a copy stream), runs the four calls and copies its result back to the
    host.  Two device input sets alternate, so step i + 1's copy runs while step i computes (the copy
    is the bound: ~210 GB/s host to device); the clock stops when the last result is on the host."""
    import torch
    names = ["draft_logits", "target_logits", "h", "last_tok"] + (["u_walk", "u_acc", "u_res"] if chain.sampled else [])
    base = chain.sets[0]
    host = {n: getattr(base, n).cpu().pin_memory() for n in names}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    dsets = chain.sets[:2]
    res_host = [(torch.empty_like(chain.acc, device="cpu").pin_memory(),
                 torch.empty_like(chain.out, device="cpu").pin_memory(),
                 torch.empty_like(chain.st, device="cpu").pin_memory()) for _ in range(2)]
    d2h = sum(t.numel() * t.element_size() for t in res_host[0])
    copy = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    t0 = None
    total = steps + 3
    for i in range(total):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        k = i % 2
        dst = dsets[k]
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(consumed[k])        # step i - 2 has finished with this set
            for n in names:
                getattr(dst, n).copy_(host[n], non_blocking=True)
            copied[k].record(copy)
        stream.wait_event(copied[k])
        chain.run(dst)
        for t_h, t_d in zip(res_host[k], (chain.acc, chain.out, chain.st)):
            t_h.copy_(t_d, non_blocking=True)
        consumed[k].record(stream)
    stream.synchronize()
    copy.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, dev, world)
    return {"value": round(whole_job_rate(shp.B, world, steps, dt), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(dt / steps * 1e3, 4),
            "pipelining": "two input sets: step i+1's host-to-device copy overlaps step i"}


# ----------------------------------------------------------- CPU oracle ----
def oracle_chain(inp, reqs, Kp=None):
    """The oracle's whole path for the requests `reqs` (first Kp positions of each)."""
    import numpy as np
    import torch

    import oracle as ref
    shp = inp.shape
    K = shp.K if Kp is None else Kp
    n = len(reqs)
    rows = np.concatenate([np.arange(b * shp.K, b * shp.K + K) for b in reqs])
    trows = np.concatenate([np.arange(b * (shp.K + 1), b * (shp.K + 1) + K + 1) for b in reqs])
    params = inp.params[reqs] if shp.temperature > 0 else None
    idx, U, lse, _ = ref.topk16(inp.draft_logits[torch.as_tensor(rows)], params=params, rows_per_param=K)
    gate = ref.ctx_gate(inp.h[torch.as_tensor(rows)], inp.Wg)
    S = ref.pair_scores(idx, U, inp.last_tok[torch.as_tensor(reqs)], inp.A, inp.Bt, gate, n, K)
    T = params["temperature"] if params is not None else np.zeros(n, np.float32)
    pt, ps, q, _ = ref.walk(idx, S, T, inp.u_walk[torch.as_tensor(reqs), :K], n, K)
    ref.verify(inp.target_logits[torch.as_tensor(trows)], pt, idx.reshape(n, K, 16), q, ps, params,
               inp.u_acc[torch.as_tensor(reqs), :K], inp.u_res[torch.as_tensor(reqs), :K + 1], n, K)


def cpu_inputs(shp, nreq):
    from dflash_draft_selection_gb300 import synth
    small = synth.Shape(**{**shp.__dict__, "B": nreq})
    return synth.make_inputs(small, device="cpu", with_conv=False)


def cpu_baseline(shp, budget_s=10.0):
    import oracle as ref
    ref.build()
    nreq = min(shp.B, 8)
    inp = cpu_inputs(shp, nreq)

    def run(budget):
        t0 = time.perf_counter()
        done = 0
        while (time.perf_counter() - t0) < budget:
            oracle_chain(inp, [done % nreq])
            done += 1
        return done, time.perf_counter() - t0

    cores = ref.num_threads()
    done, dt = run(budget_s)
    ref.set_num_threads(1)  # the same oracle on one thread, for scale
    try:
        done1, dt1 = run(budget_s / 2)
    finally:
        ref.set_num_threads(cores)
    return {"value": round(done / dt, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "value_1_thread": round(done1 / dt1, 3),
            "sample": f"{done} request chains ({nreq} distinct requests of the {shp.name} workload, K={shp.K}, "
                      f"V={shp.V}) through the whole oracle path, one after another, {dt:.1f} s "
                      f"(and {done1} on one thread in {dt1:.1f} s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle as ref
    from dflash_draft_selection_gb300 import synth
    ref.build()
    shp = synth.WORKLOADS[args.config]
    inp = cpu_inputs(shp, 2)
    t0 = time.perf_counter()
    oracle_chain(inp, [0])
    t_req = time.perf_counter() - t0
    budget = 150.0
    total = args.steps + args.warmup
    # each step is a bounded sample: the first Kp positions of one request
    Kp = shp.K
    if total * t_req > budget:
        Kp = max(1, min(shp.K, int(shp.K * budget / (total * t_req))))
    for i in range(args.warmup):
        oracle_chain(inp, [i % 2], Kp)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_chain(inp, [i % 2], Kp)
    dt = time.perf_counter() - t0
    blocks = args.steps * Kp / shp.K
    value = blocks / dt
    sample = (f"per step: positions 0..{Kp - 1} of one request of the {shp.name} workload "
              f"({Kp}/{shp.K} of a block) through the whole oracle path")
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": args.config, "B": shp.B, "K": shp.K, "V": shp.V, "hidden": shp.hidden},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "kind": "oracle", "cores": ref.num_threads(),
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
