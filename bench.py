#!/usr/bin/env python
"""Benchmark: ms per 16k-token THD pack of MiniMax-M3 MSA block-sparse attention
(prologue + index select + sparse attention forward + backward) on one GB300.

Workload: one KV group on a 16,384-token pack of 4 sequences (seeded lengths,
multiples of 128, each >= 1024), 16 query / 1 KV / 1 index head, D 128, block
128, top-16; synthetic N(0,1) bf16 inputs with per-block index-key offsets.
A step = msa_qk_norm_rope4 -> msa_index_select -> msa_sparse_attn_fwd ->
msa_sparse_attn_bwd over one pack.  Each step reads its own copy of the
inputs from a pool larger than L2, so every step starts L2-cold.

Prints one JSON line (kept short: summaries of every leg, numbers rounded;
`--detail PATH` writes the full record to a file).  Also measured in the same
run: the decode step on the paged-cache workload (B = 64, 64 q / 4 kv heads),
the end-to-end time through the public API with host buffers, the other
prefill workloads, the narrow-block variant, the CPU oracle on a bounded
sample (one core and every host core) with a parity report of sampled rows,
and per-kernel CUDA-event timings (library tracing) for the roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per 16k-token pack (index select + sparse attn fwd/bwd); TFLOP/s, % BF16 peak"
PAGES_CONTEXT = {
    "note": "the pages' own GB300 Triton timings (16k pack, 16 q / 1 kv head, D 128, block 128; "
            "pack composition unstated): attention fwd+bwd 6.7 ms, indexer select 0.62 ms",
    "fwd_bwd_ms": 6.7, "select_ms": 0.62,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--pool", type=int, default=8, help="input copies cycled through")
    ap.add_argument("--cpu-sample-tokens", type=int, default=2048)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prologue-bwd", action="store_true")
    ap.add_argument("--no-qsa", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the 64-head 16k prefill and the 32k training pack")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the oracle comparison of sampled rows in the CPU leg")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="reference arm: seconds its warm-up + timed steps may take")
    ap.add_argument("--detail", default=None, help="also write the full record here")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(seed: int, rank: int, j: int = 0) -> int:
    """Seed of input copy j on `rank`: every rank draws its own packs (weak scaling)."""
    return seed + 1000 * rank + j


def slowest_rank_ms(ms_local: float, world: int, device=None) -> float:
    """Max over ranks of a per-rank time: the job ends with its slowest rank."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_ms_per_pack(ms_step_max: float, world: int) -> float:
    """Whole-job value of the metric: `world` packs complete every ms_step_max."""
    return ms_step_max / world


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ line helpers

NOMINAL_BF16_TFLOPS = 2250.0      # GB300 dense bf16, datasheet (context only)
NOMINAL_HBM_GBS = 8000.0          # GB300 HBM3e, about 8 TB/s (context only)


def config_dict(shape, pool: int, world: int) -> dict:
    """The workload the line is quoted on; both arms print the same dict."""
    return {"workload": shape.name, "tokens": shape.T, "seqlens": list(shape.seqlens),
            "hq": shape.hq, "hkv": shape.hkv, "hi": shape.hi, "d": 128, "block": 128,
            "topk": 16,
            "step": "qk_norm_rope4 + index_select + sparse_attn_fwd + sparse_attn_bwd",
            "l2": f"inputs > L2: each GPU step reads its own copy from a {pool}-pack pool "
                  f"({pool * 144} MB)",
            "parallelism": f"replicas x{world} (one pack per GPU, no collective)"}


def rnd(x, sig: int = 4):
    """x with `sig` significant digits (recursively through dicts and lists)."""
    if isinstance(x, dict):
        return {k: rnd(v, sig) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [rnd(v, sig) for v in x]
    if isinstance(x, float):
        if x == 0 or x != x or x in (float("inf"), float("-inf")):
            return x
        from math import floor, log10
        return round(x, sig - 1 - int(floor(log10(abs(x)))))
    return x


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle arm: rank 0 alone times the oracle on every host core (a
    process per core; oracle/cpu_sample.py) and returns its JSON line; the
    other ranks return None without work."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import workloads as W
    budget = getattr(args, "ref_budget_s", 150.0)
    r = subprocess.run([sys.executable, "-m", "oracle.cpu_sample", "--mode", "reference",
                        "--config", "1", "--seed", str(args.seed), "--steps", str(args.steps),
                        "--warmup", str(args.warmup), "--budget-s", str(budget)],
                       cwd=ROOT, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle reference run failed:\n{r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    ms = res["ms_per_pack"]
    shape = W.config(1, args.seed)
    sample = (f"every query token of the pack per step (prologue rows, select, fwd, bwd), "
              f"dealt over {res['cores']} worker processes"
              if not res["scaled"] else
              f"{res['tokens_per_step']} of the pack's {res['tokens']} query tokens per step "
              f"(evenly strided; prologue rows, select, fwd, bwd) over {res['cores']} worker "
              f"processes, scaled by T/{res['tokens_per_step']}")
    line = {
        "impl": "reference", "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_dict(shape, getattr(args, "pool", 8), args.gpus),
        "cpu_baseline": {"value": ms, "unit": "ms", "cores": res["cores"], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


# ------------------------------------------------------------------ our arm

def kernel_source_hash(name: str) -> str:
    files = {"sparse_bwd_kernel": "sparse_bwd.cu", "sparse_fwd_kernel": "sparse_fwd.cu",
             "index_select_kernel": "index_select.cu", "prologue_kernel": "prologue.cu",
             "prologue_bwd_kernel": "prologue.cu",
             "decode_score_kernel": "decode.cu",
             "qsa_fwd_kernel": "qsa.cu", "qsa_bwd_dq_kernel": "qsa.cu",
             "qsa_bwd_dkv_kernel": "qsa.cu"}
    f = files.get(name)
    if f is None:
        return ""
    h = hashlib.sha256()
    for p in (os.path.join(ROOT, "msa_block_sparse_gb300", "csrc", f),
              os.path.join(ROOT, "msa_block_sparse_gb300", "csrc", "sm100_ptx.cuh")):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(name: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(name)
    if not d or d.get("source_hash") != kernel_source_hash(name):
        return None
    return d.get("bytes_per_launch")


# Kernels of the two timed phases: prefill = msa_index_select + msa_sparse_attn_fwd,
# backward = msa_sparse_attn_bwd (whose accumulator clearing is a memset, not a kernel).
PREFILL_KERNELS = ("select_plan_kernel", "index_select_kernel", "plan_kernel", "fwd_union_kernel",
                   "sparse_fwd_kernel")
BACKWARD_KERNELS = ("bwd_delta_kernel", "bwd_lists_kernel", "sparse_bwd_kernel",
                    "bwd_convert_kernel")


def phase_ms(per_step: dict, names) -> float:
    return sum(per_step.get(n, 0.0) for n in names)


def phase_pass(step_fn, nsteps, stream):
    """Runs `nsteps` steps with CUDA events only at the phase boundaries (before
    the select call, between the forward and backward calls, after the
    backward call): each phase's time then includes its memsets, launch gaps
    and the overlap of its own kernels.  step_fn(i, marks) records marks[0..2].
    Returns (prefill ms, backward ms or None) per step."""
    import torch
    marks = []
    for i in range(nsteps):
        mk = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        step_fn(i, mk)
        marks.append(mk)
    torch.cuda.synchronize()
    pf = sum(mk[0].elapsed_time(mk[1]) for mk in marks) / nsteps
    bw = sum(mk[1].elapsed_time(mk[2]) for mk in marks) / nsteps
    return pf, bw


class SideClear:
    """Clears the backward's workspace accumulators on a second stream while
    the forward runs (msa_sparse_attn_bwd_prepare), ordered after the step's
    index select (and so after the previous step's backward) and before this
    step's backward (prepared=True)."""

    def __init__(self, dev):
        import torch
        # high priority: the clear's blocks go ahead of the forward's once it
        # has started, instead of waiting behind its persistent blocks
        self.stream = torch.cuda.Stream(dev, priority=-1)
        self.after = torch.cuda.Event()
        self.cleared = torch.cuda.Event()

    def start(self, m, q, k, cu, max_seqlen, workspace):
        import torch
        self.after.record(torch.cuda.current_stream())
        self.stream.wait_event(self.after)
        m.msa_sparse_attn_bwd_prepare(q, k, cu, max_seqlen, workspace, stream=self.stream)
        self.cleared.record(self.stream)

    def join(self):
        import torch
        torch.cuda.current_stream().wait_event(self.cleared)


def time_pack(m, W, workmodel, shape, dev, stream, seed, nsteps, with_bwd, peak, sample=None):
    """Prologue + select + forward (+ backward) on one pack (inputs larger than
    L2, drawn on the CPU from `seed` so the oracle can redraw them); untimed
    warm-up, CUDA events over `nsteps`, then an event-bracketed pass for the
    per-kernel split.  `sample`: packed token ids whose selections are returned
    for the parity report."""
    import torch
    x = {k: v.to(dev) for k, v in
         W.make_prefill(shape, seed=seed, device="cpu", with_grad_out=with_bwd).items()}
    T, S, hq, hkv, hi, L = shape.T, shape.S, shape.hq, shape.hkv, shape.hi, shape.max_seqlen
    bf = torch.bfloat16
    b = {n: torch.empty((T, h, 128), dtype=bf, device=dev)
         for n, h in (("q", hq), ("k", hkv), ("qi", hi), ("ki", hi), ("o", hq))}
    sel = torch.empty((T, hi, 16), dtype=torch.int32, device=dev)
    lse = torch.empty((T, hq), dtype=torch.float32, device=dev)
    ws = {c: torch.empty(m.workspace_bytes(c, *a), dtype=torch.uint8, device=dev)
          for c, a in (("index_select", (T, S, hi, L)), ("sparse_attn_fwd", (T, S, hq, hkv, L)),
                       ("sparse_attn_bwd", (T, S, hq, hkv, L)))
          if with_bwd or c != "sparse_attn_bwd"}
    if with_bwd:
        g = {n: torch.empty_like(b[r]) for n, r in (("dq", "q"), ("dk", "k"), ("dv", "k"))}
        side = SideClear(dev)

    def step(marks=None):
        m.msa_qk_norm_rope4(x["q"], x["k"], x["q_idx"], x["k_idx"], x["w_q"], x["w_k"],
                            x["w_qi"], x["w_ki"], x["cu_seqlens"],
                            outs=(b["q"], b["k"], b["qi"], b["ki"]))
        if marks:
            marks[0].record(stream)
        m.msa_index_select(b["qi"], b["ki"], x["cu_seqlens"], L, out=sel,
                           workspace=ws["index_select"])
        if with_bwd:
            side.start(m, b["q"], b["k"], x["cu_seqlens"], L, ws["sparse_attn_bwd"])
        m.msa_sparse_attn_fwd(b["q"], b["k"], x["v"], sel, x["cu_seqlens"], L, out=b["o"],
                              lse=lse, workspace=ws["sparse_attn_fwd"])
        if marks:
            marks[1].record(stream)
        if with_bwd:
            side.join()
            m.msa_sparse_attn_bwd(b["q"], b["k"], x["v"], b["o"], x["do"], lse, sel,
                                  x["cu_seqlens"], L, dq=g["dq"], dk=g["dk"], dv=g["dv"],
                                  workspace=ws["sparse_attn_bwd"], prepared=True)
        if marks:
            marks[2].record(stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(nsteps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    pf_ms, bw_ms = phase_pass(lambda i, mk: step(mk), nsteps, stream)
    m.msa_trace_begin()
    for _ in range(nsteps):
        step()
    torch.cuda.synchronize(dev)
    tr = m.msa_trace_end()
    m.msa_check_status(dev)
    ms = e0.elapsed_time(e1) / nsteps
    wk = workmodel.prefill_work(shape.seqlens, hq, hkv, hi)
    per = {n: v["ms"] / nsteps for n, v in tr.items()}          # ms per step
    flops = wk["fwd_flops"] + wk["select_flops"] + (wk["bwd_flops"] if with_bwd else 0.0)
    out = {"workload": shape.name, "seqlens": list(shape.seqlens), "hq": hq, "hkv": hkv,
           "hi": hi, "ms_per_step": ms,
           "step": "qk_norm_rope4 + index_select + sparse_attn_fwd" +
                   (" + sparse_attn_bwd" if with_bwd else ""),
           "useful_tflops": flops / (ms * 1e-3) / 1e12, "kernels_ms": per, "work": wk}
    pf = pf_ms
    f = wk["fwd_flops"] + wk["select_flops"]
    out["prefill"] = {"ms": pf, "tflops": f / (pf * 1e-3) / 1e12,
                      "frac": f / (pf * 1e-3) / 1e12 / peak,
                      "kernels_sum_ms": phase_ms(per, PREFILL_KERNELS),
                      "kernels": list(PREFILL_KERNELS)}
    if with_bwd:
        t = per.get("sparse_bwd_kernel", 0.0)
        tb = bw_ms
        out["backward"] = {"ms": tb, "tflops": wk["bwd_flops"] / (tb * 1e-3) / 1e12,
                           "frac": wk["bwd_flops"] / (tb * 1e-3) / 1e12 / peak,
                           "kernels_sum_ms": phase_ms(per, BACKWARD_KERNELS),
                           "kernel_ms": t,
                           "kernel_frac": wk["bwd_flops"] / (t * 1e-3) / 1e12 / peak}
    if sample is not None:
        out["sample_sel"] = sel[torch.as_tensor(sample, device=dev)].cpu().numpy()
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__ as ge
    ge.build()
    import msa_block_sparse_gb300 as m
    from msa_block_sparse_gb300 import workmodel
    import workloads as W

    peaks, peak_src = load_peaks()
    parity_arrays = {}             # CUDA-path outputs of sampled rows, for the oracle
    shape = W.config(1, args.seed)
    T, S = shape.T, shape.S
    hq, hkv, hi, maxL = shape.hq, shape.hkv, shape.hi, shape.max_seqlen

    # ---- input pool (each rank draws its own pack: weak scaling)
    # pack 0 is drawn on the CPU (the oracle redraws it for the parity report),
    # the others on the device
    pool = []
    for j in range(args.pool):
        if j == 0:
            pool.append({k: v.to(dev) for k, v in
                         W.make_prefill(shape, seed=rank_seed(args.seed, rank, j), device="cpu",
                                        with_grad_out=True).items()})
        else:
            pool.append(W.make_prefill(shape, seed=rank_seed(args.seed, rank, j), device=dev,
                                       with_grad_out=True))
    cu = pool[0]["cu_seqlens"]
    bf = torch.bfloat16
    work = {
        "q": torch.empty((T, hq, 128), dtype=bf, device=dev),
        "k": torch.empty((T, hkv, 128), dtype=bf, device=dev),
        "qi": torch.empty((T, hi, 128), dtype=bf, device=dev),
        "ki": torch.empty((T, hi, 128), dtype=bf, device=dev),
        "sel": torch.empty((T, hi, 16), dtype=torch.int32, device=dev),
        "o": torch.empty((T, hq, 128), dtype=bf, device=dev),
        "lse": torch.empty((T, hq), dtype=torch.float32, device=dev),
        "dq": torch.empty((T, hq, 128), dtype=bf, device=dev),
        "dk": torch.empty((T, hkv, 128), dtype=bf, device=dev),
        "dv": torch.empty((T, hkv, 128), dtype=bf, device=dev),
    }
    ws = {c: torch.empty(max(256, m.workspace_bytes(*a)), dtype=torch.uint8, device=dev)
          for c, a in (("index_select", ("index_select", T, S, hi, maxL)),
                       ("fwd", ("sparse_attn_fwd", T, S, hq, hkv, maxL)),
                       ("bwd", ("sparse_attn_bwd", T, S, hq, hkv, maxL)))}

    side = SideClear(dev)

    def step(x, res=None, marks=None):
        res = work if res is None else res          # where o, dq, dk, dv go
        m.msa_qk_norm_rope4(x["q"], x["k"], x["q_idx"], x["k_idx"], x["w_q"], x["w_k"],
                            x["w_qi"], x["w_ki"], x["cu_seqlens"],
                            outs=(work["q"], work["k"], work["qi"], work["ki"]))
        if marks:
            marks[0].record(torch.cuda.current_stream())
        m.msa_index_select(work["qi"], work["ki"], x["cu_seqlens"], maxL, out=work["sel"],
                           workspace=ws["index_select"])
        side.start(m, work["q"], work["k"], x["cu_seqlens"], maxL, ws["bwd"])
        m.msa_sparse_attn_fwd(work["q"], work["k"], x["v"], work["sel"], x["cu_seqlens"], maxL,
                              out=res["o"], lse=work["lse"], workspace=ws["fwd"])
        if marks:
            marks[1].record(torch.cuda.current_stream())
        side.join()
        m.msa_sparse_attn_bwd(work["q"], work["k"], x["v"], res["o"], x["do"], work["lse"],
                              work["sel"], x["cu_seqlens"], maxL, dq=res["dq"], dk=res["dk"],
                              dv=res["dv"], workspace=ws["bwd"], prepared=True)
        if marks:
            marks[2].record(torch.cuda.current_stream())

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        step(pool[i % args.pool])
    torch.cuda.synchronize(dev)
    m.msa_check_status(dev)

    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    h0 = time.perf_counter()
    for i in range(args.steps):
        step(pool[i % args.pool])
    host_ms = (time.perf_counter() - h0) * 1e3 / args.steps
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    pf_ms, bw_ms = phase_pass(lambda i, mk: step(pool[i % args.pool], marks=mk), args.steps,
                              stream)
    # per-kernel times: the same steps again, every launch bracketed by CUDA
    # events on its stream (the events sit between kernels and keep each launch
    # from overlapping its predecessor's tail, so this pass is not the step time)
    m.msa_trace_begin()
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for i in range(args.steps):
        step(pool[i % args.pool])
    ev3.record(stream)
    torch.cuda.synchronize(dev)
    trace = m.msa_trace_end()
    barrier()
    clocks = sampler.stop()
    m.msa_check_status(dev)
    ms_step = ev0.elapsed_time(ev1) / args.steps
    ms_step_traced = ev2.elapsed_time(ev3) / args.steps
    ms_step = slowest_rank_ms(ms_step, world, dev)

    wk = workmodel.prefill_work(shape.seqlens, hq, hkv, hi)
    total_flops = wk["fwd_flops"] + wk["bwd_flops"] + wk["select_flops"]
    kernels = {n: {"launches": v["launches"] // args.steps if v["launches"] >= args.steps else v["launches"],
                   "ms_per_launch": v["ms"] / max(1, v["launches"]),
                   "share": None}
               for n, v in trace.items()}
    tot_ms = sum(v["ms"] for v in trace.values())
    for n, v in trace.items():
        kernels[n]["share"] = v["ms"] / tot_ms if tot_ms > 0 else None
    gpu_launches = int(sum(v["launches"] for v in trace.values()))

    flops_of = {"sparse_bwd_kernel": wk["bwd_flops"], "sparse_fwd_kernel": wk["fwd_flops"],
                "index_select_kernel": wk["select_flops"]}
    # the timed region lasts tens of milliseconds at full SM clock (sampled
    # below), so the tensor roofline is the measured burst bf16 peak; the
    # sustained (power-capped, seconds-long) figure is kept beside it
    burst = peaks.get("bf16_tflops", 1900.0)
    sustained = peaks.get("bf16_tflops_sustained", 1700.0)
    hbm = peaks.get("hbm_gbs", 6800.0)
    dom = max(trace.items(), key=lambda kv: kv[1]["ms"])[0]
    roofline = None
    if dom in flops_of:
        ms_launch = trace[dom]["ms"] / trace[dom]["launches"]
        ach = flops_of[dom] / (ms_launch * 1e-3) / 1e12
        roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": burst,
                    "unit": "TFLOP/s", "frac": ach / burst, "traffic": traffic_for(dom),
                    "peak_source": f"{peak_src} bf16 burst: {ms_step * args.steps:.0f} ms "
                                   f"timed at the sampled clock",
                    "frac_of_sustained": ach / sustained,
                    "frac_of_nominal": ach / NOMINAL_BF16_TFLOPS,
                    "flops_per_launch": flops_of[dom], "ms_per_launch": ms_launch}
    per_kernel_roofline = {}
    for n, f in flops_of.items():
        if n in trace:
            msl = trace[n]["ms"] / trace[n]["launches"]
            per_kernel_roofline[n] = {"tflops": f / (msl * 1e-3) / 1e12, "ms": msl,
                                      "frac": f / (msl * 1e-3) / 1e12 / burst}
    if "prologue_kernel" in trace:
        msl = trace["prologue_kernel"]["ms"] / trace["prologue_kernel"]["launches"]
        per_kernel_roofline["prologue_kernel"] = {
            "gbs": wk["prologue_bytes"] / (msl * 1e-3) / 1e9, "ms": msl,
            "frac": wk["prologue_bytes"] / (msl * 1e-3) / 1e9 / hbm,
            "frac_of_nominal": wk["prologue_bytes"] / (msl * 1e-3) / 1e9 / NOMINAL_HBM_GBS}
    per_step = {n: v["ms"] / args.steps for n, v in trace.items()}
    # phase times from the phase-boundary events (memsets and launch gaps
    # included); the traced kernels' sum is kept beside them
    pf, tb = slowest_rank_ms(pf_ms, world, dev), slowest_rank_ms(bw_ms, world, dev)
    pflops = wk["fwd_flops"] + wk["select_flops"]
    phases = {"prefill": {"ms": pf, "tflops": pflops / (pf * 1e-3) / 1e12,
                          "frac": pflops / (pf * 1e-3) / 1e12 / burst,
                          "kernels_sum_ms": phase_ms(per_step, PREFILL_KERNELS),
                          "kernels": list(PREFILL_KERNELS),
                          "calls": ["msa_index_select", "msa_sparse_attn_fwd"]},
              "backward": {"ms": tb, "tflops": wk["bwd_flops"] / (tb * 1e-3) / 1e12,
                           "frac": wk["bwd_flops"] / (tb * 1e-3) / 1e12 / burst,
                           "kernels_sum_ms": phase_ms(per_step, BACKWARD_KERNELS),
                           "kernels": list(BACKWARD_KERNELS),
                           "calls": ["msa_sparse_attn_bwd"]}}

    out = {
        "metric": METRIC,
        "value": job_ms_per_pack(ms_step, world),
        "unit": "ms",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_dict(shape, args.pool, world),
        "tflops": total_flops / (ms_step * 1e-3) / 1e12,
        "tokens_per_s": T * world / (ms_step * 1e-3),
        "work": wk,
        "roofline": roofline,
        "kernels": kernels,
        "kernels_pass": {"what": "a second pass of the same steps with every launch "
                                 "bracketed by CUDA events", "ms_per_step": ms_step_traced},
        "host_enqueue_ms_per_step": host_ms,
        "kernel_roofline": per_kernel_roofline,
        "phases": phases,
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "pages_context": PAGES_CONTEXT,
    }

    # ---- end to end through the public API with host buffers.  Three streams:
    # step i's inputs go up (pinned host -> device) while step i - 1 computes
    # and step i - 2's results come down; inputs and outputs are double
    # buffered on the device.  Every step still carries its own copies.
    if not args.no_e2e:
        host_in = {k: v.cpu().pin_memory() for k, v in pool[0].items()}
        out_names = ("o", "dq", "dk", "dv")
        dev_in = [{k: torch.empty_like(v) for k, v in pool[0].items()} for _ in range(2)]
        dev_out = [{n: torch.empty_like(work[n]) for n in out_names} for _ in range(2)]
        host_out = [{n: torch.empty(work[n].shape, dtype=work[n].dtype).pin_memory()
                     for n in out_names} for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        up_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n, first=None):
            """n pipelined steps; `first` is recorded on the upload stream first."""
            if first is not None:
                first.record(s_up)
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(s_up):
                    if i >= 2:
                        s_up.wait_event(in_free[b])
                    for k in host_in:
                        dev_in[b][k].copy_(host_in[k], non_blocking=True)
                    up_done[b].record(s_up)
                stream.wait_event(up_done[b])
                if i >= 2:
                    stream.wait_event(down_done[b])
                step(dev_in[b], dev_out[b])
                in_free[b].record(stream)
                comp_done[b].record(stream)
                with torch.cuda.stream(s_down):
                    s_down.wait_event(comp_done[b])
                    for nme in out_names:
                        host_out[b][nme].copy_(dev_out[b][nme], non_blocking=True)
                    down_done[b].record(s_down)

        e2e_steps(3)
        torch.cuda.synchronize(dev)
        # as many steps as the device-resident timing, so that the unoverlapped
        # first upload and last download weigh as little as in a long job
        n_e2e = max(5, args.steps)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps(n_e2e, first=e0)
        e1.record(s_down)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = slowest_rank_ms(e0.elapsed_time(e1) / n_e2e, world, dev)
        out["e2e"] = {"value": job_ms_per_pack(e2e_ms, world), "unit": "ms",
                      "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "steps": n_e2e,
                      "schedule": "upload, compute and download on three streams, "
                                  "double-buffered; each step includes its own copies"}

    # ---- prologue backward (q and k of the same pack): dx, dw from x and dy
    if not args.no_prologue_bwd:
        gen = torch.Generator(device=dev).manual_seed(args.seed + 77)
        dyk = [torch.randn((T, hkv, 128), generator=gen, device=dev).to(torch.bfloat16)
               for _ in range(args.pool)]
        dxq = torch.empty((T, hq, 128), dtype=torch.bfloat16, device=dev)
        dxk = torch.empty((T, hkv, 128), dtype=torch.bfloat16, device=dev)
        dwq = torch.empty(128, dtype=torch.float32, device=dev)
        dwk = torch.empty(128, dtype=torch.float32, device=dev)
        pws = torch.empty(m.workspace_bytes("qk_norm_rope_bwd", T, hq), dtype=torch.uint8,
                          device=dev)

        def pstep(i):
            x = pool[i % args.pool]
            m.msa_qk_norm_rope_bwd(x["q"], x["do"], x["w_q"], x["cu_seqlens"], dx=dxq, dw=dwq,
                                   workspace=pws)
            m.msa_qk_norm_rope_bwd(x["k"], dyk[i % args.pool], x["w_k"], x["cu_seqlens"],
                                   dx=dxk, dw=dwk, workspace=pws)

        for i in range(3):
            pstep(i)
        torch.cuda.synchronize(dev)
        npb = max(10, args.steps)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for i in range(npb):
            pstep(i)
        p1.record(stream)
        torch.cuda.synchronize(dev)
        m.msa_trace_begin()          # per-kernel times from a second, event-bracketed pass
        for i in range(npb):
            pstep(i)
        torch.cuda.synchronize(dev)
        ptrace = m.msa_trace_end()
        m.msa_check_status(dev)
        pms = p0.elapsed_time(p1) / npb
        pbytes = 3 * 2 * T * (hq + hkv) * 128          # x, dy read; dx written (bf16)
        pgbs = pbytes / (pms * 1e-3) / 1e9
        out["prologue_bwd"] = {
            "workload": f"{shape.name}: q ({hq} heads) and k ({hkv})", "ms_per_step": pms,
            "gbs": pgbs, "bytes_per_step": pbytes,
            "roofline": {"bound": "hbm", "achieved": pgbs, "peak": peaks.get("hbm_gbs", 6800.0),
                         "unit": "GB/s", "frac": pgbs / peaks.get("hbm_gbs", 6800.0),
                         "traffic": traffic_for("prologue_bwd_kernel"),
                         "peak_source": f"{peak_src} HBM copy"},
            "kernels": {n: {"launches": v["launches"] // npb, "ms_per_launch": v["ms"] / v["launches"]}
                        for n, v in ptrace.items()},
        }

    # ---- decode step on the paged-cache workload
    if not args.no_decode:
        dshape = W.config(3, args.seed)
        dx = W.make_decode(dshape, seed=rank_seed(args.seed, rank), device=dev)
        B, maxp = dshape.B, dx["block_table"].shape[1]
        dws = torch.empty(m.workspace_bytes("decode_step", B, dshape.hq, dshape.hkv, maxp),
                          dtype=torch.uint8, device=dev)
        od = torch.empty_like(dx["q"])
        sd = torch.empty((B, dshape.hkv, 16), dtype=torch.int32, device=dev)

        def dstep():
            m.msa_decode_step(dx["q"], dx["q_idx"], dx["k_cache"], dx["v_cache"], dx["kidx_cache"],
                              dx["block_table"], dx["cache_lens"], out=od, sel_out=sd,
                              workspace=dws)

        for _ in range(3):
            dstep()
        torch.cuda.synchronize(dev)
        nd = max(10, args.steps)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(nd):
            dstep()
        d1.record(stream)
        torch.cuda.synchronize(dev)
        m.msa_trace_begin()          # per-kernel times from a second, event-bracketed pass
        for _ in range(nd):
            dstep()
        torch.cuda.synchronize(dev)
        dtrace = m.msa_trace_end()
        m.msa_check_status(dev)
        dms = d0.elapsed_time(d1) / nd
        # parity rows (two shortest caches and the longest): their pages as bf16
        # bits, the GPU's selection and output, before the append below writes
        # new tokens into the caches
        if not args.no_parity and rank == 0 and world == 1:
            import numpy as np
            lens_np = dx["cache_lens"].cpu().numpy()
            rows = sorted(set(np.argsort(lens_np)[:2].tolist() + [int(np.argmax(lens_np))]))
            table_np = dx["block_table"].cpu().numpy()
            used = sorted({int(p_) for r_ in rows for p_ in table_np[r_, :(lens_np[r_] + 127) // 128]})
            remap = {p_: i for i, p_ in enumerate(used)}
            sub = np.full((len(rows), table_np.shape[1]), -1, dtype=np.int64)
            for n_, r_ in enumerate(rows):
                for c_ in range((lens_np[r_] + 127) // 128):
                    sub[n_, c_] = remap[int(table_np[r_, c_])]
            idx = torch.tensor(used, dtype=torch.long, device=dev)
            bits = lambda t: t.index_select(0, idx).view(torch.int16).cpu().numpy()   # noqa: E731
            ridx = torch.tensor(rows, dtype=torch.long, device=dev)
            parity_arrays.update(
                dec_name=np.array(dshape.name), dec_rows=np.array(rows),
                dec_q=dx["q"][ridx].float().cpu().numpy(),
                dec_q_idx=dx["q_idx"][ridx].float().cpu().numpy(),
                dec_k_bits=bits(dx["k_cache"]), dec_v_bits=bits(dx["v_cache"]),
                dec_kidx_bits=bits(dx["kidx_cache"]), dec_table=sub, dec_lens=lens_np[rows],
                dec_sel=sd[ridx].cpu().numpy(), dec_o=od[ridx].float().cpu().numpy())
        # the decode append (prologue of the new tokens, written into their pages)
        # on the same caches, timed on its own
        agen = torch.Generator(device=dev).manual_seed(args.seed + 5)
        araw = {n: torch.randn((B, h, 128), generator=agen, device=dev).to(torch.bfloat16)
                for n, h in (("q", dshape.hq), ("q_idx", dshape.hkv), ("k", dshape.hkv),
                             ("v", dshape.hkv), ("k_idx", dshape.hkv))}
        aw = {n: (torch.randn(128, generator=agen, device=dev) * 0.2).to(torch.bfloat16)
              for n in ("w_q", "w_qi", "w_k", "w_ki")}
        aq, aqi = torch.empty_like(dx["q"]), torch.empty_like(dx["q_idx"])

        def astep():
            m.msa_decode_append(araw["q"], araw["q_idx"], araw["k"], araw["v"], araw["k_idx"],
                                aw["w_q"], aw["w_qi"], aw["w_k"], aw["w_ki"], dx["k_cache"],
                                dx["v_cache"], dx["kidx_cache"], dx["block_table"],
                                dx["cache_lens"], q_out=aq, q_idx_out=aqi)

        for _ in range(3):
            astep()
        torch.cuda.synchronize(dev)
        # one call is a few microseconds of GPU work, less than the binding's
        # host-side checks: time ten calls captured in a CUDA graph instead
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for _ in range(10):
                    astep()
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        reps = max(3, nd // 10)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            graph.replay()
        a1.record(stream)
        torch.cuda.synchronize(dev)
        m.msa_check_status(dev)
        ams = a0.elapsed_time(a1) / (10 * reps)
        dbytes = workmodel.decode_bytes(dshape.cache_lens, dshape.hq, dshape.hkv)
        gbs = dbytes / (dms * 1e-3) / 1e9
        out["decode"] = {
            "workload": dshape.name, "batch": B, "ms_per_step": dms,
            "gbs": gbs, "bytes_per_step": dbytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks.get("hbm_gbs", 6800.0),
                         "unit": "GB/s", "frac": gbs / peaks.get("hbm_gbs", 6800.0),
                         "traffic": traffic_for("decode_score_kernel"),
                         "peak_source": f"{peak_src} HBM copy"},
            "kernels": {n: {"launches": v["launches"] // nd, "ms_per_launch": v["ms"] / v["launches"]}
                        for n, v in dtrace.items()},
            "l2": "the index-key cache (%.2f GB) is larger than L2" %
                  (dx["kidx_cache"].numel() * 2 / 1e9),
            "append": {"ms_per_step": ams, "kernel": "decode_append_kernel",
                       "what": "prologue of B new tokens (q, index-q; k, index-k, v into "
                               "their pages), timed on its own from a CUDA graph of ten "
                               "calls"},
        }
        del dx

    # ---- the other prefill workloads: full layer shape on a 16k pack (prefill)
    # and the 32k training pack (prefill + backward)
    if not args.no_configs:
        import numpy as np
        out["configs"] = {}
        for key, idx, nsteps, with_bwd in (("cfg2", 2, 10, False), ("cfg4", 4, 5, True)):
            cshape = W.config(idx, args.seed)
            cseed = rank_seed(args.seed, rank)
            samp = np.sort(np.random.default_rng(100 + idx).choice(cshape.T, 512, replace=False))
            r_ = time_pack(m, W, workmodel, cshape, dev, stream, cseed, nsteps, with_bwd, burst,
                           sample=samp)
            parity_arrays.update({f"{key}_tokens": samp, f"{key}_sel": r_.pop("sample_sel"),
                                  f"{key}_seed": np.array(cseed)})
            out["configs"][cshape.name] = r_

    # ---- narrow-block variant: 16k pack, 12 q / 1 kv heads, head dim 256, 4-token
    # blocks, fwd + bwd (the pages' second timed workload)
    if not args.no_qsa:
        qshape = W.qsa_config(1, args.seed)
        qx = W.make_qsa(qshape, seed=rank_seed(args.seed, rank), device=dev)
        qcu, qL = qx["cu_seqlens"], qshape.max_seqlen
        qo = torch.empty_like(qx["q"])
        qlse = torch.empty((qshape.T, qshape.hq), dtype=torch.float32, device=dev)
        qdq, qdk, qdv = torch.empty_like(qx["q"]), torch.empty_like(qx["k"]), torch.empty_like(qx["v"])
        qws_f = torch.empty(m.workspace_bytes("qsa_attn_fwd", qshape.T, qshape.S, qshape.hq,
                                              qshape.hkv, qL), dtype=torch.uint8, device=dev)
        qws_b = torch.empty(m.workspace_bytes("qsa_attn_bwd", qshape.T, qshape.S, qshape.hq,
                                              qshape.hkv, qL), dtype=torch.uint8, device=dev)

        def qstep():
            m.msa_qsa_attn_fwd(qx["q"], qx["k"], qx["v"], qx["sel"], qcu, qL, out=qo, lse=qlse,
                               workspace=qws_f)
            m.msa_qsa_attn_bwd(qx["q"], qx["k"], qx["v"], qo, qx["do"], qlse, qx["sel"], qcu, qL,
                               dq=qdq, dk=qdk, dv=qdv, workspace=qws_b)

        for _ in range(3):
            qstep()
        torch.cuda.synchronize(dev)
        nq = max(5, min(args.steps, 20))
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for _ in range(nq):
            qstep()
        q1.record(stream)
        torch.cuda.synchronize(dev)
        m.msa_trace_begin()          # per-kernel times from a second, event-bracketed pass
        for _ in range(nq):
            qstep()
        torch.cuda.synchronize(dev)
        qtrace = m.msa_trace_end()
        m.msa_check_status(dev)
        qms = q0.elapsed_time(q1) / nq
        qwk = workmodel.qsa_work(qshape.seqlens, qx["sel"].cpu().numpy(), qshape.hq)
        qflops = qwk["fwd_flops"] + qwk["bwd_flops"]
        qk = {n: {"launches": v["launches"] // nq, "ms_per_launch": v["ms"] / v["launches"]}
              for n, v in qtrace.items()}
        qkr = {}
        for n, f in (("qsa_fwd_kernel", qwk["fwd_flops"]),
                     ("qsa_bwd_dq_kernel", qwk["bwd_flops"] * 3 / 5),
                     ("qsa_bwd_dkv_kernel", qwk["bwd_flops"] * 2 / 5)):
            if n in qk:
                t = qk[n]["ms_per_launch"]
                qkr[n] = {"ms": t, "useful_tflops": f / (t * 1e-3) / 1e12,
                          "frac": f / (t * 1e-3) / 1e12 / burst, "traffic": traffic_for(n)}
        out["qsa"] = {
            "workload": qshape.name, "seqlens": list(qshape.seqlens), "hq": qshape.hq,
            "hkv": qshape.hkv, "d": W.QSA_D, "block": W.QSA_BLOCK, "topk": qshape.topk,
            "ms_per_step": qms, "step": "msa_qsa_attn_fwd + msa_qsa_attn_bwd",
            "useful_tflops": qflops / (qms * 1e-3) / 1e12,
            "frac": qflops / (qms * 1e-3) / 1e12 / burst,
            "work": qwk, "kernels": qk, "kernel_roofline": qkr,
            "useful_split": "dq pass: S, dP, dQ = 3 of the 5 backward products; dkv pass: "
                            "dV, dK = 2 of 5 (each pass also recomputes S and dP)",
            "l2": "q, dO, o (100 MB each) and the fp32 accumulators exceed L2",
            "pages_context": {"fwd_bwd_ms": 16.4, "note": "the pages' GB300 Triton time for "
                              "this workload shape (pack composition and selection unstated)"},
        }
        del qx

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only): one core and
    # every host core, and the parity report of sampled rows.  The CUDA
    # path's outputs go to the oracle process in a temporary .npz.
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        import shutil
        import tempfile

        import numpy as np
        cmd = [sys.executable, "-m", "oracle.cpu_sample", "--mode", "baseline", "--config", "1",
               "--tokens", str(args.cpu_sample_tokens), "--seed", str(rank_seed(args.seed, 0, 0))]
        tmpdir = None
        if not args.no_parity:
            step(pool[0])                       # pack 0: drawn on the CPU, redrawn by the oracle
            torch.cuda.synchronize(dev)
            m.msa_check_status(dev)
            toks = np.sort(np.random.default_rng(0).choice(T, size=min(args.cpu_sample_tokens, T),
                                                           replace=False))
            ti = torch.as_tensor(toks, device=dev)
            parity_arrays.update(cfg1_tokens=toks, cfg1_sel=work["sel"][ti].cpu().numpy(),
                                 cfg1_o=work["o"][ti].float().cpu().numpy(),
                                 cfg1_lse=work["lse"][ti].cpu().numpy(),
                                 cfg1_dq=work["dq"][ti].float().cpu().numpy())
            tmpdir = tempfile.mkdtemp(prefix="msa_parity_")
            path = os.path.join(tmpdir, "gpu_outputs.npz")
            np.savez(path, **parity_arrays)
            cmd += ["--parity", path]
        try:
            r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=1200)
        finally:
            if tmpdir:
                shutil.rmtree(tmpdir, ignore_errors=True)
        if r.returncode == 0:
            cs = json.loads(r.stdout.strip().splitlines()[-1])
            out["cpu_baseline"] = {
                "value": cs["ms_per_pack"], "unit": "ms", "cores": cs["cores"], "kind": "oracle",
                "sample": f"prologue+select+fwd+bwd of {cs['sample_tokens']} random tokens of "
                          f"pack 0 over {cs['cores']} processes, x T/{cs['sample_tokens']}",
                "one_core": {"value": cs["ms_per_pack_1core"], "cores": 1},
                "seconds_1core": {k: cs[k] for k in ("prologue_s", "select_s", "fwd_s", "bwd_s")}}
            if "parity" in cs:
                out["parity"] = cs["parity"]
        else:
            out["cpu_baseline"] = {"value": None, "error": r.stderr[-800:]}

    if rank == 0:
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump(out, f, indent=1, default=str)
        print(json.dumps(compact_line(out)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def compact_line(out: dict) -> dict:
    """The printed line: the contract's keys, then short summaries of every
    leg (full detail: --detail)."""
    keep = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
            "e2e", "gpu_launches", "clocks", "cpu_baseline")
    line = {k: out[k] for k in keep if k in out}
    if line.get("roofline"):
        line["roofline"] = {k: v for k, v in line["roofline"].items()
                            if k not in ("flops_per_launch", "ms_per_launch")}
    if line.get("cpu_baseline"):
        line["cpu_baseline"] = {k: v for k, v in line["cpu_baseline"].items()
                                if k != "seconds_1core"}
    if line.get("e2e"):
        line["e2e"] = {k: v for k, v in line["e2e"].items() if k not in ("schedule", "steps")}
    line["tflops"] = out.get("tflops")
    short = lambda n: n[:-len("_kernel")] if n.endswith("_kernel") else n   # noqa: E731
    line["phases"] = {k: {"ms": v["ms"], "tflops": v["tflops"], "frac": v["frac"]}
                      for k, v in out.get("phases", {}).items()}
    line["kernels_ms"] = {short(n): v["launches"] * v["ms_per_launch"]       # per step
                          for n, v in out.get("kernels", {}).items()}
    line["kernel_frac"] = {short(n): v["frac"] for n, v in out.get("kernel_roofline", {}).items()}
    if "decode" in out:
        d = out["decode"]
        line["decode"] = {"ms": d["ms_per_step"], "gbs": d["gbs"], "frac": d["roofline"]["frac"],
                          "frac_of_nominal": d["gbs"] / NOMINAL_HBM_GBS,
                          "score_ms": d["kernels"].get("decode_score_kernel", {}).get("ms_per_launch"),
                          "append_ms": d["append"]["ms_per_step"]}
    if "prologue_bwd" in out:
        d = out["prologue_bwd"]
        line["prologue_bwd"] = {"ms": d["ms_per_step"], "frac": d["roofline"]["frac"]}
    if "configs" in out:
        line["configs"] = {}
        for name, c in out["configs"].items():
            e = {"ms": c["ms_per_step"], "prefill_ms": c["prefill"]["ms"],
                 "prefill_frac": c["prefill"]["frac"]}
            if "backward" in c:
                e.update(bwd_ms=c["backward"]["ms"], bwd_frac=c["backward"]["frac"],
                         bwd_kernel_frac=c["backward"]["kernel_frac"])
            line["configs"][name] = e
    if "qsa" in out:
        qd = out["qsa"]
        line["qsa"] = {"ms": qd["ms_per_step"], "tflops": qd["useful_tflops"], "frac": qd["frac"],
                       "kernel_frac": {short(n): v["frac"] for n, v in qd["kernel_roofline"].items()}}
    if "parity" in out:
        line["parity"] = {n: {k: v for k, v in p.items()} for n, p in out["parity"].items()}
    return rnd(line)


def main():
    args = parse()
    if args.impl == "reference":
        line = run_reference(args)
        if line is not None:
            print(json.dumps(line), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
