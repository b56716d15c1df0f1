#!/usr/bin/env python
"""Benchmark of the packed native-resolution attention hot path on B300.

One step = the whole path over one synthetic pack: mf_pack_plan (device
scan, per-token ids, RoPE table), mf_attn_fwd and mf_attn_bwd (forward-only
workloads: plan and forward).  Throughput is
reported as fwd+bwd TFLOP/s with FLOPs = 4*heads*head_dim*sum(L_i^2) forward
and 2.5x that backward (algorithmic: only the per-sample blocks count).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mf|reference]

N > 1 runs under torchrun: every rank plans and runs its own pack (same
shapes, its own tensor values) -- packs are independent, so there is no
exchange and scaling is weak.  Rank 0 prints one JSON line.

`--impl reference` times the float64 CPU oracle (the only CPU code this
benchmark may run) on bounded samples of the same workload.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed 2D-RoPE varlen attention fwd+bwd TFLOP/s; fraction of bf16 TC peak"
METRIC_FWD = "packed 2D-RoPE varlen attention fwd TFLOP/s; fraction of bf16 TC peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mf", "reference"], default="mf")
    ap.add_argument("--mode", choices=["step", "cfg", "chain"], default="step",
                    help="step: the fwd+bwd training step (the headline); cfg: the CFG pair pack's "
                         "packed forward + guidance against two separate forwards; chain: one attention "
                         "block's memory-bound chains fused against unfused")
    ap.add_argument("--guidance", type=float, default=4.0)
    ap.add_argument("--workload", default="native_res_32k", choices=list(synth.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-threads", type=int, default=0, help="BLAS threads of the oracle baseline (0: all)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    return ap.parse_args()


def sample_len(smp):
    """Tokens of one (text_len, height_px, width_px[, frames]) sample."""
    frames = smp[3] if len(smp) > 3 else 1
    return smp[0] + frames * (smp[1] // 16) * (smp[2] // 16)


def pack_flops(samples, heads, head_dim):
    lens = [sample_len(s) for s in samples]
    s2 = float(sum(L * L for L in lens))
    fwd = 4.0 * heads * head_dim * s2
    return fwd, 2.5 * fwd, lens


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.path = None
        self.gpu_id = None
        try:
            u = torch.cuda.get_device_properties(device).uuid
            self.gpu_id = "GPU-" + str(u)
        except Exception:
            self.gpu_id = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# oracle (CPU) baseline
# --------------------------------------------------------------------------

_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "OMP_NUM_THREADS")


def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return int(max(i.get("num_threads", 1) for i in info)) if info else 1
    except Exception:
        for var in _BLAS_ENV:
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return os.cpu_count() or 1


def oracle_sample(wl, seconds, max_heads=None, threads=0):
    """Time the oracle's fwd+bwd on one sample of the workload, head after
    head, until `seconds` of CPU work (or all heads) are done; `threads` > 0
    caps the BLAS threads (0: all of them)."""
    if threads > 0:
        try:
            import threadpoolctl
        except ImportError:
            # without threadpoolctl the BLAS pool is sized at start-up only
            if _blas_threads() != threads:
                raise SystemExit(f"--cpu-threads {threads}: start with " +
                                 " ".join(f"{v}={threads}" for v in _BLAS_ENV) + " (threadpoolctl is missing)")
            return oracle_sample(wl, seconds, max_heads)
        with threadpoolctl.threadpool_limits(limits=threads):
            return oracle_sample(wl, seconds, max_heads)
    import oracle
    lens = [sample_len(s) for s in wl.samples]
    # the sample whose length is closest to 3,600 tokens: large enough to be
    # representative, small enough that one head takes about a second
    si = int(np.argmin([abs(L - 3600) for L in lens]))
    s = wl.samples[si]
    p = oracle.pack_plan([s])
    n = p["total_tokens"]
    g = torch.Generator("cpu").manual_seed(wl.seed)
    shape = (n, 1, wl.head_dim)
    heads = 0
    flop = 0.0
    t0 = time.perf_counter()
    while True:
        q, k, v, do = (torch.randn(shape, generator=g).to(torch.bfloat16).double().numpy() for _ in range(4))
        rope = dict(frame=p["frame"], rope_axes=wl.rope_axes)
        O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"], **rope)
        oracle.attn_bwd(q, k, v, O, L, do, p["cu_seqlens"], p["pos"], **rope)
        heads += 1
        flop += 3.5 * 4.0 * wl.head_dim * n * n
        el = time.perf_counter() - t0
        if el >= seconds or heads >= (max_heads or wl.heads):
            break
    return {"value": flop / el / 1e12, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "seconds": round(el, 3),
            "sample": f"float64 oracle fwd+bwd of sample {si} ({n} tokens) of the {wl.name} pack, "
                      f"{heads} head(s) x head_dim {wl.head_dim}"}


# --------------------------------------------------------------------------
# multi-rank host logic (N > 1 under torchrun; tested with gloo on CPU)
# --------------------------------------------------------------------------

def rank_workload(wl, rank):
    """Rank `rank`'s pack: the same shapes as `wl`, its own tensor values."""
    return synth.Workload(wl.name, wl.samples, wl.heads, wl.head_dim, wl.passes, wl.token_budget,
                          wl.cfg_pairs, seed=wl.seed + 1000 * rank)


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest `x` over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, step_flop, ms_step):
    """Whole-job throughput: every rank's step FLOPs over the slowest rank's time."""
    return world * step_flop / (ms_step * 1e-3) / 1e12


# --------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# --------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    wl = synth.WORKLOADS[args.workload](args.seed)
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0, max_heads=1)
    t0 = time.perf_counter()
    vals = []
    last = None
    for _ in range(args.steps):
        last = oracle_sample(wl, 0.0, max_heads=1)
        vals.append(last["value"])
    el = time.perf_counter() - t0
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{wl.name} seed {wl.seed}", "step": last["sample"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# the library arm
# --------------------------------------------------------------------------

def run_mf(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import packed_resolution_diffusion_plan_b300 as mf

    wl = synth.WORKLOADS[args.workload](args.seed)
    fwd_flop, bwd_flop, lens = pack_flops(wl.samples, wl.heads, wl.head_dim)
    # Forward-only workloads (the single 1024^2 image, the CFG pair pack) time
    # plan + forward; the training packs time plan + forward + backward.
    fwd_only = wl.passes == "fwd"
    if fwd_only:
        bwd_flop = 0.0
    step_flop = fwd_flop + bwd_flop
    host = synth.draw_tensors(rank_workload(wl, rank), with_grad=True)
    T, H, D = host["q"].shape
    q, k, v, do = (host[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(mf.bwd_workspace_bytes(T, H, D), dtype=torch.uint8, device=dev)
    ws_fwd = torch.empty(mf.fwd_workspace_bytes(T, H, D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def backward(q, k, v, o, lse, do, plan, ws, dq, dk, dv, stream=None):
        mf.attn_bwd(q, k, v, o, lse, do, plan, workspace=ws, dq=dq, dk=dk, dv=dv, stream=stream)

    def step(ev=None):
        plan = mf.pack_plan(wl.samples, token_budget=wl.token_budget, head_dim=D, device=dev,
                            rope_axes=wl.rope_axes)
        if ev is not None:
            mf.record_main_kernel(ev[0], ev[1])
        mf.attn_fwd(q, k, v, plan, out=o, lse=lse, workspace=ws_fwd)
        if fwd_only:
            return plan
        if ev is not None:
            mf.record_main_kernel(ev[2], ev[3])
        backward(q, k, v, o, lse, do, plan, ws, dq, dk, dv)
        return plan

    # Each step plans anew, and every plan carries its own status word: check
    # them all, so that a timeout in any step fails the run.
    for _ in range(max(args.warmup, 1)):
        plan = step()
        mf.check(plan)
    launches_per_step = 3 + 2 + (0 if fwd_only else 3)  # scan, ids, RoPE table; fwd pre, main; bwd pre, main, dq

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A step whose tensors fit in L2 twice over (the single 1024^2 image:
    # ~0.16 GB with the rotated copies) is timed step by step with a 512 MB
    # write between steps, outside the timed spans, so that no step finds the
    # previous one's data in L2; larger packs stream more than L2 per step.
    step_bytes = T * H * D * 2 * (4 if fwd_only else 9)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if step_bytes < 2 * 126e6 else None
    spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)] if flush is not None else None
    clocks = ClockSampler(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start.record(stream)
    plans = []
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
            spans[i][0].record(stream)
        plans.append(step(evs[i]))
        if flush is not None:
            spans[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    for plan in plans:
        mf.check(plan)
    if flush is not None:
        ms_step = float(np.sum([a.elapsed_time(b) for a, b in spans])) / args.steps
    else:
        ms_step = t_start.elapsed_time(t_end) / args.steps
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    bwd_main_ms = None if fwd_only else float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    ms_step = max_over_ranks(ms_step, dist, dev)
    value = job_tflops(world, step_flop, ms_step)

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs in from pinned host memory and its results (O, LSE,
    # dQ, dK, dV) back out.  Steps run as a pipeline over three streams and two
    # device buffer sets: step i+1's input copies and step i-1's result copies
    # overlap step i's plan + forward + backward; events keep a buffer set
    # from being overwritten before the step that uses it is done.
    in_names = ("q", "k", "v") if fwd_only else ("q", "k", "v", "do")
    out_names = ("o",) if fwd_only else ("o", "dq", "dk", "dv")
    pin = {n: host[n].pin_memory() for n in in_names}
    out_h = {n: torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory() for n in out_names}
    lse_h = torch.empty((H, T), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in out_h.values()) + lse_h.numel() * 4
    sets = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws, wsf=ws_fwd)]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    e2e_plans = []

    def e2e_step(i):
        j = i % 2
        b = sets[j]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[j])  # step i-2 has finished reading these inputs
            for n in in_names:
                b[n].copy_(pin[n], non_blocking=True)
            ev_in[j].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev_in[j])
            if i >= 2:
                s_cmp.wait_event(ev_out[j])  # step i-2's results have left these buffers
            p = mf.pack_plan(wl.samples, token_budget=wl.token_budget, head_dim=D, device=dev,
                             rope_axes=wl.rope_axes, stream=s_cmp)
            mf.attn_fwd(b["q"], b["k"], b["v"], p, out=b["o"], lse=b["lse"], workspace=b["wsf"], stream=s_cmp)
            if not fwd_only:
                backward(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], p, b["ws"],
                         b["dq"], b["dk"], b["dv"], stream=s_cmp)
            ev_cmp[j].record(s_cmp)
            e2e_plans.append(p)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[j])
            for n in out_names:
                out_h[n].copy_(b[n], non_blocking=True)
            lse_h.copy_(b["lse"], non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(s_in)
    for i in range(args.e2e_steps):
        e2e_step(2 + i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    for p in e2e_plans:
        mf.check(p)
    mf.check(plan)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    # The timed region is a burst of well under a second, so the denominator
    # is the burst bf16 figure; the sustained one (seconds of back-to-back
    # GEMMs under the power cap) is reported beside it.
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    kernels = {"attn_fwd_kernel": {"ms": fwd_ms, "flop": fwd_flop}}
    if not fwd_only:
        kernels["bwd_main_kernel"] = {"ms": bwd_main_ms, "flop": bwd_flop}
    for kname, kd in kernels.items():
        kd["tflops"] = kd["flop"] / (kd["ms"] * 1e-3) / 1e12
        kd["frac_burst"] = kd["tflops"] / peak
        kd["frac_sustained"] = kd["tflops"] / peak_sustained
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    traffic = load_traffic(dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": kernels[dom]["tflops"], "peak": peak,
                "unit": "TFLOP/s", "frac": kernels[dom]["tflops"] / peak, "traffic": traffic,
                "peak_kind": f"bf16_tflops, burst ({peak_src})",
                "frac_of_sustained_peak": kernels[dom]["tflops"] / peak_sustained,
                "step_frac": value / world / peak,
                "per_kernel": {n: {k2: round(v2, 4) for k2, v2 in kd.items()} for n, kd in kernels.items()}}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(wl, args.cpu_seconds, threads=args.cpu_threads)
    line = {
        "metric": METRIC_FWD if fwd_only else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "precision": "bf16 inputs/outputs; tcgen05 MMAs with fp32 accumulation (logit products on fp16 "
                     "rotated Q/K rows, P*V and dO products in bf16)",
        "config": {"workload": f"{wl.name} seed {wl.seed}", "samples": [list(x) for x in wl.samples],
                   "seq_lens": lens, "total_tokens": T, "heads": H, "head_dim": D,
                   "token_budget": wl.token_budget, "fwd_tflop": fwd_flop / 1e12, "bwd_tflop": bwd_flop / 1e12,
                   "step": "pack plan + forward" if fwd_only else "pack plan + forward + backward",
                   "l2": (f"flushed: a 512 MB write between timed steps (Q/K/V/O are {T * H * D * 2 / 1e6:.0f} MB "
                          "each), each step timed on its own" if flush is not None else
                          f"no flush: Q/K/V/dO/O are {T * H * D * 2 / 1e6:.0f} MB each (> 126 MB L2)"),
                   "parallelism": f"{world} independent pack(s), one per GPU"},
        "tokens_per_s": world * T / (ms_step * 1e-3),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(world, step_flop, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "per step: inputs in from pinned host memory, plan + fwd + bwd, all results out; "
                            "step i+1's and i-1's copies overlap step i's compute (3 streams, 2 buffer sets)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if wl.name.endswith("_padded"):
        # the packed pack's own work, done inside the padded batch's time
        base = synth.WORKLOADS[wl.name[:-len("_padded")]](args.seed)
        uf, ub, ulens = pack_flops(base.samples, base.heads, base.head_dim)
        line["padding"] = {"packed_workload": base.name, "packed_tokens": int(sum(ulens)),
                           "padded_tokens": T, "useful_tflops": job_tflops(world, uf + ub, ms_step),
                           "note": "value counts the padded batch's work; useful_tflops counts only "
                                   "the packed samples' work over the same time"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd.cu", "attn_common.cuh", "ptx.cuh", "common.cuh"],
    "bwd_main_kernel": ["attn_bwd.cu", "attn_common.cuh", "ptx.cuh", "common.cuh"],
}


_CODE_TOKENS = None


def code_only(text):
    """C++/CUDA source without its comments, whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps the hash."""
    import re
    global _CODE_TOKENS
    if _CODE_TOKENS is None:
        _CODE_TOKENS = re.compile(r'("(?:\\.|[^"\\])*")|/\*.*?\*/|//[^\n]*', re.S)
    text = _CODE_TOKENS.sub(lambda m: m.group(1) or " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel, root=None):
    """Hash of the code (comments excluded) of the files `kernel` is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(root or ROOT, "packed_resolution_diffusion_plan_b300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel):
    """DRAM bytes per launch of `kernel` from its committed ncu summary
    (profiles/<kernel>_traffic.txt), or None when there is none or when the
    kernel's sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                key, val = line.split(":", 1)
                fields[key.strip()] = val.strip()
    if fields.get("source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return float(fields["bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_cfg(args):
    """Inference with classifier-free guidance on the CFG pair pack (4 prompts at
    1024^2, conditional and unconditional branches): one packed forward of both
    branches followed by the guidance, against two separate forwards (the
    conditional samples, then the unconditional ones).  The guidance kernel does
    the same work either way and is timed once, on the packed output."""
    import packed_resolution_diffusion_plan_b300 as mf
    dev = torch.device("cuda", 0)
    wl = synth.cfg_pair(args.seed)
    host = synth.draw_tensors(wl, with_grad=False)
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    T, H, D = q.shape
    segs = wl.segments()
    starts = np.concatenate([[0], np.cumsum([a + b for a, b in segs])]).astype(int)
    cond_idx = [i for i in range(len(segs)) if i % 2 == 0]
    unc_idx = [i for i in range(len(segs)) if i % 2 == 1]

    def gather(idx):
        rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in idx])
        r = torch.as_tensor(rows, device=dev)
        return [x.index_select(0, r).contiguous() for x in (q, k, v)]

    qc, kc, vc = gather(cond_idx)
    qu, ku, vu = gather(unc_idx)
    plan = mf.pack_plan(wl.samples, head_dim=D)
    plan_c = mf.pack_plan([wl.samples[i] for i in cond_idx], head_dim=D)
    plan_u = mf.pack_plan([wl.samples[i] for i in unc_idx], head_dim=D)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    oc, lc = torch.empty_like(qc), torch.empty((H, qc.shape[0]), dtype=torch.float32, device=dev)
    ou, lu = torch.empty_like(qu), torch.empty((H, qu.shape[0]), dtype=torch.float32, device=dev)
    ws = torch.empty(mf.fwd_workspace_bytes(T, H, D), dtype=torch.uint8, device=dev)
    guided = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def packed():
        mf.attn_fwd(q, k, v, plan, out=o, lse=lse, workspace=ws)

    def separate():
        mf.attn_fwd(qc, kc, vc, plan_c, out=oc, lse=lc, workspace=ws)
        mf.attn_fwd(qu, ku, vu, plan_u, out=ou, lse=lu, workspace=ws)

    def combine():
        mf.cfg_combine(o, plan, args.guidance, out=guided)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(dev)
    clocks.start()
    t_packed = timed(packed)
    t_sep = timed(separate)
    t_comb = timed(combine)
    clk = clocks.stop()
    for p in (plan, plan_c, plan_u):
        mf.check(p)
    fwd_flop, _, lens = pack_flops(wl.samples, H, D)
    line = {"metric": "CFG inference: packed cond+uncond attention forward + guidance, speedup over two "
                      "separate forwards + guidance",
            "value": (t_sep + t_comb) / (t_packed + t_comb), "unit": "x", "higher_is_better": True,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{wl.name} seed {wl.seed}", "total_tokens": T, "heads": H, "head_dim": D,
                       "guidance": args.guidance},
            "packed_fwd_ms": t_packed, "separate_fwd_ms": t_sep, "combine_ms": t_comb,
            "packed_fwd_tflops": fwd_flop / (t_packed * 1e-3) / 1e12,
            "gpu_launches": 2 * args.steps + 4 * args.steps + args.steps,
            "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


def run_chain(args):
    """One joint-attention block forward on a pack (synthetic weights, hidden =
    heads * head_dim): x -> LN + modulation -> @W_qkv -> attention -> @W_o ->
    gate + residual.  Fused: mf_norm_modulate, mf_attn_fwd_qkv (split + RoPE in
    its first pass), mf_gate_residual.  Unfused: the same operations as
    separate torch kernels (layer_norm, gather of the per-sample vectors, mul,
    add, contiguous q/k/v copies, mf_attn_fwd, mul, add).  Both use the same
    cuBLAS products and the same attention kernel; the JSON line reports each
    part and the memory-bound chains' total both ways."""
    import packed_resolution_diffusion_plan_b300 as mf
    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS[args.workload](args.seed)
    H, D = wl.heads, wl.head_dim
    C = H * D
    plan = mf.pack_plan(wl.samples, token_budget=wl.token_budget, head_dim=D, device=dev, rope_axes=wl.rope_axes)
    T, n = plan.total_tokens, plan.n_samples
    g = torch.Generator("cpu").manual_seed(args.seed)

    def rnd(*shape, scale=1.0):
        return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).to(dev)

    x = rnd(T, C)
    w_qkv, w_o = rnd(C, 3 * C, scale=C ** -0.5), rnd(C, C, scale=C ** -0.5)
    shift, scale, gate = rnd(n, C, scale=0.2), rnd(n, C, scale=0.2), rnd(n, C, scale=0.5)
    sample_of = torch.repeat_interleave(torch.arange(n, device=dev), torch.diff(plan.cu_seqlens().long()))
    ws = torch.empty(mf.fwd_workspace_bytes(T, H, D), dtype=torch.uint8, device=dev)
    y, z, out = torch.empty_like(x), torch.empty((T, C), dtype=torch.bfloat16, device=dev), torch.empty_like(x)
    qkv = torch.empty((T, 3 * C), dtype=torch.bfloat16, device=dev)
    o = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = {}

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(name, []).append(e)

    def fused():
        mark("f0"); mf.norm_modulate(x, plan, shift, scale, out=y)
        mark("f1"); torch.matmul(y, w_qkv, out=qkv)
        mark("f2"); mf.record_main_kernel(*main_ev["f"]); mf.attn_fwd_qkv(qkv, plan, H, out=o, lse=lse, workspace=ws)
        mark("f3"); torch.matmul(o.view(T, C), w_o, out=z)
        mark("f4"); mf.gate_residual(x, z, plan, gate, out=out)
        mark("f5")

    def unfused():
        mark("u0")
        yn = torch.nn.functional.layer_norm(x, (C,), eps=1e-6)
        yu = yn * (1 + scale.index_select(0, sample_of)) + shift.index_select(0, sample_of)
        mark("u1"); q3 = torch.matmul(yu, w_qkv)
        mark("u2")
        q, k, v = (q3[:, i * C:(i + 1) * C].contiguous().view(T, H, D) for i in range(3))
        mf.record_main_kernel(*main_ev["u"]); mf.attn_fwd(q, k, v, plan, out=o, lse=lse, workspace=ws)
        mark("u3"); zz = torch.matmul(o.view(T, C), w_o)
        mark("u4"); _ = x + gate.index_select(0, sample_of) * zz
        mark("u5")

    main_ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in "fu"}
    for _ in range(max(args.warmup, 3)):
        fused(); unfused()
    torch.cuda.synchronize(dev)
    ev.clear()
    mains = {"f": [], "u": []}
    clocks = ClockSampler(dev)
    clocks.start()
    for _ in range(args.steps):
        fused(); unfused()
        torch.cuda.synchronize(dev)
        for k2 in "fu":
            mains[k2].append(main_ev[k2][0].elapsed_time(main_ev[k2][1]))
    clk = clocks.stop()
    mf.check(plan)

    def span(a, b):
        return float(np.median([ea.elapsed_time(eb) for ea, eb in zip(ev[a], ev[b])]))

    f = {"norm_modulate": span("f0", "f1"), "qkv_gemm": span("f1", "f2"), "attention": span("f2", "f3"),
         "out_gemm": span("f3", "f4"), "gate_residual": span("f4", "f5")}
    u = {"norm_modulate": span("u0", "u1"), "qkv_gemm": span("u1", "u2"), "attention": span("u2", "u3"),
         "out_gemm": span("u3", "u4"), "gate_residual": span("u4", "u5")}
    fm, um = float(np.median(mains["f"])), float(np.median(mains["u"]))
    # memory-bound chains: everything but the two products and the attention main kernel
    f_chain = f["norm_modulate"] + (f["attention"] - fm) + f["gate_residual"]
    u_chain = u["norm_modulate"] + (u["attention"] - um) + u["gate_residual"]
    f_block, u_block = sum(f.values()), sum(u.values())
    line = {"metric": "joint-attention block forward: fused memory-bound chains (norm + modulation, QKV split + "
                      "RoPE, gate + residual) against the same operations unfused",
            "value": u_chain / f_chain, "unit": "x (chain time, unfused / fused)", "higher_is_better": True,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
            "data": "synthetic (random weights)",
            "config": {"workload": f"{wl.name} seed {wl.seed}", "total_tokens": T, "hidden": C, "heads": H,
                       "head_dim": D},
            "fused_ms": {k2: round(v2, 4) for k2, v2 in f.items()},
            "unfused_ms": {k2: round(v2, 4) for k2, v2 in u.items()},
            "attention_main_kernel_ms": round(fm, 4),
            "chain_ms": {"fused": round(f_chain, 4), "unfused": round(u_chain, 4)},
            "block_ms": {"fused": round(f_block, 4), "unfused": round(u_block, 4)},
            "block_speedup": u_block / f_block,
            # x read, y written; k read, k~ written (q is rotated from the QKV rows
            # inside the attention kernel); x, z read, out written
            "chain_hbm_gbs_fused": (2 * T * C * 2 + 2 * T * C * 2 + 3 * T * C * 2) / (f_chain * 1e-3) / 1e9,
            "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "cfg":
        return run_cfg(args)
    if args.mode == "chain":
        return run_chain(args)
    return run_mf(args)


if __name__ == "__main__":
    sys.exit(main())
