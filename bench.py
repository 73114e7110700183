"""Benchmark of the MoE expert block on GB300.

A step is one pass of the whole block (counts -> fc1 + SwiGLU -> fc2 +
weighted combine) over one workload, inputs already in HBM.  The headline
workload is ``skew``, the largest one that fits one GPU (T=16384 tokens,
H=2048, I=768, E=128 experts, top-8, W=8 logical ranks, bf16, Zipf(1.2)
routing).  L2 is flushed (a 256 MB write) between timed steps, outside the
timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

With no --workload it prints one full JSON line for each of the context
workloads (tiny, decode, uniform, int8) and then the headline skew line,
last; with --workload, that workload's line only.  N > 1 (under torchrun)
runs one independent replica per GPU (weak scaling): the block has no
exchange step on one GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_dispatch_histc_gb300.workloads import WORKLOADS, as_f64, make_inputs  # noqa: E402

METRIC = "MoE expert-block tokens/s (1 GPU); grouped-GEMM TFLOP/s as fraction of GB300 bf16 peak"
PROFILE_DIR = os.path.join(ROOT, "profiles")
GMM_SRC = os.path.join(ROOT, "moe_expert_dispatch_histc_gb300", "csrc", "gmm.cu")
GMMQ_SRC = os.path.join(ROOT, "moe_expert_dispatch_histc_gb300", "csrc", "gmm_q.cu")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _src_hash(path):
    """Hash of a source file's code: comments and blank space removed, so an
    edit of comments alone keeps the recorded counters valid."""
    import re
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = "\n".join(l.strip() for l in src.splitlines() if l.strip())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def _ncu_traffic(kernel_key, workload, src=GMM_SRC):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current source of the kernel's file; else None."""
    p = os.path.join(PROFILE_DIR, "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel_key}:{workload}")
    if not ent or ent.get("src_sha256_16") != _src_hash(src):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _oracle_sample(wl, inp):
    """A callable running the oracle on tokens [a, a + n) of the workload."""
    from oracle import mc2_oracle as orc
    if wl.act == "i8":
        def run(a, n):
            orc.quant_block_forward(inp["x"][a:a + n], inp["xs"][a:a + n], inp["w1"], inp["w1s"],
                                    inp["w2"], inp["w2s"], inp["sel"][a:a + n],
                                    inp["probs"][a:a + n], wl.E, wl.W)
        return run
    x = as_f64(inp["x"], wl.act)
    w1 = as_f64(inp["w1"], wl.act)
    w2 = as_f64(inp["w2"], wl.act)

    def run(a, n):
        orc.block_forward(x[a:a + n], w1, w2, inp["sel"][a:a + n], inp["probs"][a:a + n],
                          wl.E, wl.W, h_dtype=wl.act)
    return run


def cpu_baseline(wl, inp, budget_s=12.0):
    """The oracle as it stands, on host cores, on the first T_s tokens of the
    same workload (all experts' weights, same routing)."""
    run = _oracle_sample(wl, inp)
    Ts, spent, done = 0, 0.0, 0
    step = max(wl.W, (256 // wl.W) * wl.W)
    while spent < budget_s and Ts < wl.T:
        n = min(step, wl.T - Ts)
        t0 = time.perf_counter()
        run(Ts, n)
        spent += time.perf_counter() - t0
        Ts += n
        done += 1
    return {"value": Ts / spent, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {Ts} of {wl.T} tokens of the {wl.name} workload in {done} chunks of "
                      f"{step} tokens (numpy oracle, float64 / int64, all experts), {spent:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = WORKLOADS[args.workload or HEADLINE]
    inp = make_inputs(wl, 0)
    run = _oracle_sample(wl, inp)
    Ts = max(wl.W, (64 // wl.W) * wl.W)   # bounded sample of the workload per step

    def step(i):
        run((i * Ts) % wl.T, Ts)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = Ts * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _headline_config(wl),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{Ts} tokens of the {wl.name} workload per step (numpy "
                                   f"oracle, float64 / int64, all experts; host memory, no L2 "
                                   f"flush)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(value: float, world: int, device="cuda") -> float:
    """The job's time of a region timed on every rank: the slowest rank's."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank's tokens over
    the slowest rank's time."""
    return tokens_per_rank * world * steps / (max_ms / 1e3)


def _headline_config(wl):
    """The config of a workload's line as the cuda arm prints it (the reference
    arm reports the same workload under the same config)."""
    c = _config(wl, l2="flushed (256 MB write) between steps")
    c["role"] = "headline" if wl.name == HEADLINE else "context (the headline line is last)"
    return c


def _config(wl, l2):
    return {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
            "W": wl.W, "act": wl.act, "routing": wl.routing, "l2": l2,
            "parallelism": "replicas" if int(os.environ.get("WORLD_SIZE", "1")) > 1 else "1gpu"}


def e2e_pipelined(wl, d, b, stream, steps, run):
    """Milliseconds of `steps` pipelined end-to-end steps (see run_cuda), and
    the bytes each step copies to and from the host."""
    import dataclasses

    import torch

    names = [n for n in ("x", "xs", "sel", "probs") if d.get(n) is not None]
    host = {n: d[n].cpu().pin_memory() for n in names}
    dev = [{n: d[n] for n in names}, {n: torch.empty_like(d[n]) for n in names}]
    outs = [b.out, torch.empty_like(b.out)]
    h_out = [torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory() for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        k = i % 2
        if i >= 2:
            s_h2d.wait_event(ev_comp[k])       # step i-2 has read set k
        with torch.cuda.stream(s_h2d):
            for n in names:
                dev[k][n].copy_(host[n], non_blocking=True)
            ev_h2d[k].record(s_h2d)
        stream.wait_event(ev_h2d[k])
        if i >= 2:
            stream.wait_event(ev_d2h[k])       # step i-2's output is back on the host
        dd = dict(d)
        dd.update(dev[k])
        run(dd, dataclasses.replace(b, out=outs[k]))
        ev_comp[k].record(stream)
        s_d2h.wait_event(ev_comp[k])
        with torch.cuda.stream(s_d2h):
            h_out[k].copy_(outs[k], non_blocking=True)
            ev_d2h[k].record(s_d2h)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_h2d.wait_event(t0)
    s_d2h.wait_event(t0)
    for i in range(steps):
        step(i)
    t1.record(s_d2h)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    bi = sum(h.numel() * h.element_size() for h in host.values())
    bo = h_out[0].numel() * h_out[0].element_size()
    return ms, bi, bo


HEADLINE = "skew"                                # the largest single-GPU workload
CONTEXT = ("tiny", "decode", "uniform", "int8")  # printed before the headline line


def run_cuda(args):
    """One JSON line per workload: with no --workload, the four context
    workloads first and the headline (skew) line last; else that workload."""
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from moe_expert_dispatch_histc_gb300 import binding as B
    from moe_expert_dispatch_histc_gb300.build import build
    build()
    B.lib()
    B.mc2_set_tile_pairing({"auto": 0, "single": 1, "pairs": 2}[args.tiling])
    names = [args.workload] if args.workload else [*CONTEXT, HEADLINE]
    if args.path == "unfused":   # the non-fused baseline exists for bf16 workloads only
        names = [n for n in names if WORKLOADS[n].act == "bf16"]
    for name in names:
        run_cuda_workload(args, WORKLOADS[name], headline=(name == HEADLINE))
        torch.cuda.empty_cache()
    if world > 1:
        dist.destroy_process_group()


def run_cuda_workload(args, wl, headline):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from moe_expert_dispatch_histc_gb300 import binding as B, block as blk
    inp = make_inputs(wl, 0)
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    shape = blk.shape_of(wl)
    stream = torch.cuda.current_stream()
    # int8 path: expand the weights to bf16 once (load-time weight transform,
    # outside the timed region; a no-op for the float paths)
    torch.cuda.synchronize()
    t_prepack = time.perf_counter()
    blk.prepack(wl, d, b, stream=stream)
    torch.cuda.synchronize()
    t_prepack = time.perf_counter() - t_prepack
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")  # 256 MB > L2

    unfused = args.path == "unfused"
    xp = None
    if unfused:
        if wl.act != "bf16":
            raise SystemExit("--path unfused: bf16 workloads only")
        xp = torch.empty(wl.R, wl.H, dtype=torch.bfloat16, device="cuda")

    def seg_counts():
        B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src,
                         b.unpermute_dst, b.ws, b.dev_status, stream=stream)

    def seg_permute():
        B.mc2_permute_rows(shape, d["x"], b.permute_src, xp, stream=stream)

    def seg_fc1():
        if unfused:
            B.mc2_gmm_swiglu(shape, xp, d["w1"], b.offsets, b.h, b.dev_status, stream=stream)
        else:
            B.mc2_alltoallv_gmm(shape, d["x"], d["xs"], d["w1"], d["w1s"], b.offsets,
                                b.permute_src, b.ws, b.h, b.h_scale, b.dev_status, stream=stream)

    def seg_fc2():
        B.mc2_gmm_alltoallv(shape, b.h, b.h_scale, d["w2"], d["w2s"], b.offsets, b.permute_src,
                            b.unpermute_dst, d["probs"], b.ws, b.out, b.dev_status, stream=stream)

    segments = [("counts", seg_counts)] + ([("permute", seg_permute)] if unfused else []) + \
        [("fc1_swiglu", seg_fc1), ("fc2_combine", seg_fc2)]
    nseg = len(segments)

    def step(kernel_events=None):
        n = 0
        for i, (name, fn) in enumerate(segments):
            timed = kernel_events is not None and name == "fc1_swiglu"
            if timed:  # events around the fc1 kernel itself, recorded by the library
                B.mc2_set_gemm_events(*kernel_events)
            try:
                fn()
            finally:
                if timed:
                    B.mc2_set_gemm_events(None, None)
            n += B.mc2_last_launch_count()
            if i + 1 < nseg:
                ev[i + 1].record(stream)
        return n

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)]
    for _ in range(args.warmup):
        flush.zero_()
        ev[0].record(stream)
        step()
        ev[nseg].record(stream)
    torch.cuda.synchronize()
    if int(b.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(b.dev_status.item())} after warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)]
              for _ in range(args.steps)]
    kevents = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in kevents:  # a first record creates the CUDA events the library records
        k[0].record(stream)
        k[1].record(stream)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    # ~1 ms of GPU-side wait before the first timed step (outside its events):
    # the host, which enqueues each segment through its own C call, gets that
    # far ahead, so no timed segment waits for the host to submit its work
    torch.cuda._sleep(2_000_000)
    launches = 0
    for i in range(args.steps):
        flush.zero_()
        ev = events[i]
        ev[0].record(stream)
        launches += step(kevents[i])
        ev[nseg].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    seg = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(nseg)]
                    for e in events])  # ms per segment, in the order of `segments`
    segi = {name: i for i, (name, _) in enumerate(segments)}
    total_ms = float(seg.sum())
    total_ms = max_over_ranks(total_ms, world)
    value = job_tokens_per_s(wl.T, world, args.steps, total_ms)

    # e2e: every step copies its inputs (x, ids, probs; int8 also the token
    # scales) from pinned host memory and reads its output back to pinned host
    # memory, through the public entry point.  The copies of step i+1 and the
    # read-back of step i-1 run on their own streams while step i computes
    # (two device sets of the per-step tensors); the timed region spans the
    # first copy to the last read-back.  No flush: the weights a step streams
    # (w1 + w2) are larger than L2.
    e2e_steps = max(3, args.steps // 4)
    if unfused:
        e2e_run = lambda dd, bb: blk.run_unfused(wl, dd, bb, xp, stream=stream)  # noqa: E731
    else:
        e2e_run = lambda dd, bb: blk.run_block(wl, dd, bb, stream=stream)  # noqa: E731
    e2e_ms, bi, bo = e2e_pipelined(wl, d, b, stream, e2e_steps, e2e_run)
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_val = job_tokens_per_s(wl.T, world, e2e_steps, e2e_ms)

    if rank != 0:
        if world > 1:
            dist.barrier()
        return
    peaks, src = _peaks()
    fc1_ms = float(seg[:, segi["fc1_swiglu"]].mean())
    # the fc1 kernel alone: CUDA events the library recorded around its launch
    fc1_kernel_ms = float(np.mean([k[0].elapsed_time(k[1]) for k in kevents]))
    fc2_ms = float(seg[:, segi["fc2_combine"]].mean())
    fc1_flops = 2 * wl.R * wl.H * 2 * wl.I
    peak = float(peaks["bf16_tflops"])
    if wl.act == "f32":   # tf32 tensor cores: the bf16 measured peak x the nominal 1.1 / 2.25
        peak *= 1.1 / 2.25
    tflops = wl.flops / ((fc1_ms + fc2_ms) / 1e3) / 1e12
    # fc1's algorithmic bytes: the weights of experts that got rows, x, h
    offs = b.offsets.cpu().numpy().astype(np.int64)
    touched = int((np.diff(offs) > 0).sum())
    esz = {"f32": 4, "bf16": 2, "i8": 1}[wl.act]
    fc1_bytes = touched * wl.H * 2 * wl.I * esz + wl.T * wl.H * esz + \
        int(offs[-1]) * wl.I * (4 if wl.act == "f32" else 2)
    hbm = float(peaks["hbm_gbs"])
    if fc1_flops / fc1_bytes < peak * 1e12 / (hbm * 1e9):   # below the ridge: bound by HBM
        roof = {"bound": "hbm", "achieved": fc1_bytes / (fc1_kernel_ms / 1e3) / 1e9, "peak": hbm,
                "unit": "GB/s", "peak_source": f"{src} hbm_gbs"}
    else:
        roof = {"bound": "tensor", "achieved": fc1_flops / (fc1_kernel_ms / 1e3) / 1e12, "peak": peak,
                "unit": "TFLOP/s",
                "peak_source": f"{src} bf16_tflops (burst)" +
                               (" x 1.1/2.25 (nominal tf32 : bf16)" if wl.act == "f32" else "")}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["algorithmic"] = {"flops": fc1_flops, "bytes": fc1_bytes}
    roof["kernel_ms"] = fc1_kernel_ms
    roof["timing"] = ("CUDA events the library records on the call's stream right before and "
                      "after the fc1 kernel's launch, every timed step")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32 (fp32 storage)" if wl.act == "f32" else "bf16",
        "data": "synthetic", "config": _config(wl, l2="flushed (256 MB write) between steps"),
        "tflops": tflops, "tflops_frac_of_peak": tflops / peak,
        "segments_ms": {name: float(seg[:, i].mean()) for name, i in segi.items()},
        "step_ms_median": float(np.median(seg.sum(axis=1))),
        "segments_ms_median": {name: float(np.median(seg[:, i])) for name, i in segi.items()},
        "roofline": {"kernel": ("gmm_kernel<fc1 rows> (fc1 + SwiGLU on materialised rows)"
                                if unfused else
                                "gmm_qw_kernel<fc1> (permute gather + exact int8 fc1 + dequant + "
                                "SwiGLU)" if wl.act == "i8" else
                                "gmm_kernel<fc1, tf32> (permute gather + fc1 + SwiGLU)"
                                if wl.act == "f32" else
                                "gmm_kernel<fc1> (permute gather + fc1 + SwiGLU)"),
                     **roof,
                     "traffic": None if unfused else
                     _ncu_traffic("gmm_fc1", wl.name, GMMQ_SRC if wl.act == "i8" else GMM_SRC)},
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "steps": e2e_steps,
                "mode": ("counts, mc2_permute_rows, mc2_gmm_swiglu, mc2_gmm_alltoallv per step"
                         if unfused else "mc2_moe_forward per step") +
                        "; the next step's host->device copies and the "
                        "previous step's device->host read-back overlap the compute (two "
                        "buffer sets, three streams); no L2 flush (w1 + w2 exceed L2)"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    # the counts step against HBM: ids read once; counts, offsets and both
    # index maps written (a few microseconds: launch and barrier latency bound)
    c_ms = line["segments_ms"]["counts"]
    R = wl.T * wl.k
    c_bytes = 4 * (R + 2 * wl.W * wl.E + wl.E + 1 + 2 * R)
    line["counts"] = {"ms": c_ms, "bytes": c_bytes, "achieved_gbs": c_bytes / (c_ms / 1e3) / 1e9,
                      "frac_of_hbm": c_bytes / (c_ms / 1e3) / 1e9 / hbm}
    if unfused:
        line["config"]["path"] = "unfused: materialised permute + plain grouped fc1"
    if args.tiling != "auto":
        line["config"]["tiling"] = args.tiling
    if wl.act == "i8":
        line["weight_prepack_ms"] = t_prepack * 1e3
        line["dtype"] = "int8 (exact, on bf16 tensor cores)"
        line["roofline"]["peak_source"] += "; int8 runs at the bf16 rate (no integer tcgen05 MMA on sm_103a)"
    if wl.name == "tiny":
        line["config"]["note"] = ("correctness only: 64 tokens, a few-microsecond block; its "
                                  "roofline fraction says nothing about the kernels")
    line["config"]["role"] = "headline" if headline else "context (the headline line is last)"
    assert headline == (wl.name == HEADLINE)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, budget_s=12.0 if headline else 6.0)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()


def run_backward(args):
    """Backward of the block (bf16): one mc2_moe_backward per step (both
    dgrads, SwiGLU backward, the unpermute-sum of dx, both weight gradients;
    G as the training forward kept it, or recomputed with --recompute-g), with
    the counts, the kept G and the transposed weights prepared once.
    Metric: tokens/s of the backward; roofline on the call's tensor work
    (12*R*H*I flops, 16*R*H*I with the recompute)."""
    import torch
    from moe_expert_dispatch_histc_gb300 import binding as B, block as blk
    from moe_expert_dispatch_histc_gb300.build import build
    build()
    B.lib()
    wl = WORKLOADS[args.workload or "uniform"]
    if wl.act != "bf16":
        raise SystemExit("--op backward: bf16 workloads only")
    inp = make_inputs(wl, 0)
    d = blk.inputs_to_device(inp, wl)
    b = blk.alloc_buffers(wl)
    shape = blk.shape_of(wl)
    stream = torch.cuda.current_stream()
    B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src, b.unpermute_dst,
                     b.ws, b.dev_status, stream=stream)
    w1t = torch.empty(wl.E, 2 * wl.I, wl.H, dtype=torch.bfloat16, device="cuda")
    w2t = torch.empty(wl.E, wl.H, wl.I, dtype=torch.bfloat16, device="cuda")
    B.mc2_transpose_weights(shape, d["w1"], d["w2"], w1t, w2t, stream=stream)
    rng = np.random.default_rng(1)
    dout_np = rng.standard_normal((wl.T, wl.H)).astype(np.float32)
    dout = torch.from_numpy(dout_np).cuda().to(torch.bfloat16)
    ws = torch.empty(B.mc2_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    g_kept = None
    if not args.recompute_g:   # the training forward keeps G; done once, outside the timing
        g_kept = torch.empty(wl.R, 2 * wl.I, dtype=torch.bfloat16, device="cuda")
        h_tmp = torch.empty(wl.R, wl.I, dtype=torch.bfloat16, device="cuda")
        B.mc2_alltoallv_gmm_keep(shape, d["x"], d["w1"], b.offsets, b.permute_src, h_tmp, g_kept,
                                 b.dev_status, stream=stream)
    dx = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device="cuda")
    dw1 = torch.empty(wl.E, wl.H, 2 * wl.I, device="cuda")
    dw2 = torch.empty(wl.E, wl.I, wl.H, device="cuda")
    dprobs = torch.empty(wl.T, wl.k, device="cuda")
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")

    def call():
        B.mc2_moe_backward(shape, d["x"], d["probs"], d["w1"], w1t, w2t, dout, b.offsets,
                           b.permute_src, b.unpermute_dst, dx, dw1, dw2, dprobs, ws,
                           b.dev_status, stream=stream, g=g_kept)
        return B.mc2_last_launch_count()
    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.2)
    evs, launches = [], 0
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launches += call()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(b.dev_status.item()) != 0:
        raise RuntimeError(f"device status {int(b.dev_status.item())}")
    ms = float(np.mean([a.elapsed_time(c) for a, c in evs]))
    value = wl.T / (ms / 1e3)
    flops = (12.0 if g_kept is not None else 16.0) * wl.R * wl.H * wl.I
    peaks, src = _peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / (ms / 1e3) / 1e12
    # end to end: x, ids, probs and dout in from pinned host memory, every step
    # (counts included: the ids arrive with the step); the gradients that leave
    # the block towards the layers before it, dx and dprobs, back to the host.
    # dw1 and dw2 stay on the device, where an optimizer step consumes them.
    host = {n: d[n].cpu().pin_memory() for n in ("x", "sel", "probs")}
    h_dout = dout.cpu().pin_memory()
    outs = [dx, dprobs]
    h_outs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    e2e_steps = max(3, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for n, h in host.items():
            d[n].copy_(h, non_blocking=True)
        dout.copy_(h_dout, non_blocking=True)
        B.mc2_moe_counts(shape, d["sel"], b.cnt, b.recv, b.offsets, b.permute_src,
                         b.unpermute_dst, b.ws, b.dev_status, stream=stream)
        call()
        for h, o in zip(h_outs, outs):
            h.copy_(o, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    bi = sum(h.numel() * h.element_size() for h in host.values()) + h_dout.numel() * 2
    bo = sum(h.numel() * h.element_size() for h in h_outs)
    # CPU oracle on a bounded sample of the same workload
    from oracle import mc2_oracle as orc
    x64, w1, w2 = (as_f64(inp[n], wl.act) for n in ("x", "w1", "w2"))
    Ts = min(wl.T, max(wl.W, (512 // wl.W) * wl.W))
    t0 = time.perf_counter()
    orc.block_backward(x64[:Ts], w1, w2, inp["sel"][:Ts], inp["probs"][:Ts],
                       dout_np[:Ts].astype(np.float64), wl.E, wl.W, h_dtype="bf16")
    cpu_s = time.perf_counter() - t0
    line = {
        "metric": "MoE expert-block backward tokens/s (1 GPU)", "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**_config(wl, l2="flushed (256 MB write) between steps"), "op": "backward",
                   "G": "recomputed" if g_kept is None else "kept by mc2_alltoallv_gmm_keep"},
        "tflops": achieved,
        "roofline": {"kernel": "the whole backward call (12*R*H*I flops of gradients, "
                               "+4*R*H*I when G is recomputed)", "bound": "tensor",
                     "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"{src} bf16_tflops (burst)", "traffic": None},
        "e2e": {"value": wl.T / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "steps": e2e_steps,
                "mode": "inputs and dout in, counts + backward, dx and dprobs out (dw1, dw2 "
                        "stay on the device), serially"},
        "cpu_baseline": {"value": Ts / cpu_s, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"first {Ts} of {wl.T} tokens, all experts (numpy float64 "
                                   f"chain rule), {cpu_s:.1f} s"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


MMRS = {"W": 8, "m": 4096, "k": 1024, "n": 4096}   # TP over 8 ranks of a K=8192 projection


def run_mmrs(args):
    """Quantised matmul + reduce-scatter over W logical ranks (one C call per
    step: int8 -> bf16 copies, then the fused CTA-pair kernel that folds every
    rank's dequantised product into an on-chip sum; --path twopass: the exact
    int8 grouped GEMM with one group per rank writing int32 partials, then the
    rank-ordered dequant + sum).  Metric: int8 tera-ops/s of the whole
    operation (2*m*W*k*n per call)."""
    import torch
    from moe_expert_dispatch_histc_gb300 import binding as B
    from moe_expert_dispatch_histc_gb300.build import build
    build()
    B.lib()
    W, m, k, n = MMRS["W"], MMRS["m"], MMRS["k"], MMRS["n"]
    twopass = args.path == "twopass"
    B.mc2_set_mmrs_path(1 if twopass else 0)
    rng = np.random.default_rng(0)
    x1 = rng.integers(-127, 128, (W, m, k)).astype(np.int8)
    x2 = rng.integers(-127, 128, (W, k, n)).astype(np.int8)
    x1s = rng.uniform(1e-3, 1e-2, (W, m)).astype(np.float32)
    x2s = rng.uniform(1e-3, 1e-2, (W, n)).astype(np.float32)
    s = B.MmrsShape(m, k, n, W)
    ws = torch.empty(B.mc2_mm_reduce_scatter_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    out = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = [torch.from_numpy(a).cuda() for a in (x1, x1s, x2, x2s)]
    stream = torch.cuda.current_stream()
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")

    def call():
        B.mc2_mm_reduce_scatter_i8(s, d[0], d[1], d[2], d[3], out, ws, st, stream=stream)
        return B.mc2_last_launch_count()
    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.2)
    evs, launches = [], 0
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launches += call()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    ops = 2.0 * m * W * k * n
    value = ops / (ms / 1e3) / 1e12
    # end to end: inputs from pinned host memory, output back, every call
    h = [t.cpu().pin_memory() for t in d]
    h_out = torch.empty(m, n, dtype=torch.bfloat16).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, args.steps // 4)
    e0.record(stream)
    for _ in range(e2e_steps):
        for dst, src in zip(d, h):
            dst.copy_(src, non_blocking=True)
        call()
        h_out.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    bi = sum(t.numel() * t.element_size() for t in h)
    # CPU oracle on a bounded sample: the first rows of every rank's block
    from oracle import mc2_oracle as orc
    ms_rows = 8 * W
    t0 = time.perf_counter()
    orc.mm_reduce_scatter(x1[:, :ms_rows], x1s[:, :ms_rows], x2, x2s)
    cpu_s = time.perf_counter() - t0
    cpu_val = 2.0 * ms_rows * W * k * n / cpu_s / 1e12
    peaks, src = _peaks()
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": "int8 matmul + reduce-scatter over logical ranks, tera-ops/s (1 GPU)",
        "value": value, "unit": "TOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 (exact, on bf16 tensor cores)", "data": "synthetic",
        "config": {"workload": f"mm_reduce_scatter W{W} m{m} k{k} n{n}", **MMRS,
                   "path": "twopass" if twopass else "fused",
                   "l2": "flushed (256 MB write) between steps"},
        "roofline": {"kernel": "the whole call (int8->bf16 copies, " +
                               ("gmm_q_kernel, mmrs_reduce_kernel)" if twopass
                                else "mmrs_fused_kernel)"),
                     "bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / peak,
                     "peak_source": f"{src} bf16_tflops (burst); int8 runs at the bf16 rate",
                     "traffic": None},
        "e2e": {"value": ops / (e2e_ms / 1e3) / 1e12, "unit": "TOP/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": m * n * 2, "steps": e2e_steps,
                "mode": "inputs copied in, call, output copied back, serially per step"},
        "cpu_baseline": {"value": cpu_val, "unit": "TOP/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"first {ms_rows} rows of each of the {W} ranks (int64 "
                                   f"numpy matmul), {cpu_s:.1f} s"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                    help="one workload; default: tiny, decode, uniform and int8 as context "
                         "lines, then the headline skew line (the largest workload) last")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="fused", choices=["fused", "unfused", "twopass"],
                    help="unfused: the non-fused baseline (materialised permute, plain grouped "
                         "fc1), bf16 workloads only; twopass (--op mm_reduce_scatter): int32 "
                         "partials through memory, then a reduce kernel")
    ap.add_argument("--tiling", default="auto", choices=["auto", "single", "pairs"],
                    help="grouped-GEMM tiling of the block (mc2_set_tile_pairing): all give "
                         "the same bits")
    ap.add_argument("--recompute-g", action="store_true",
                    help="--op backward: recompute G instead of taking the training forward's")
    ap.add_argument("--op", default="block", choices=["block", "backward", "mm_reduce_scatter"],
                    help="mm_reduce_scatter: the quantised matmul + reduce-scatter over "
                         "logical ranks (a separate line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.path == "twopass" and args.op != "mm_reduce_scatter":
        ap.error("--path twopass goes with --op mm_reduce_scatter")
    if args.op == "mm_reduce_scatter" and args.path == "unfused":
        ap.error("--op mm_reduce_scatter takes --path fused or twopass")
    if args.op == "backward":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--op backward has its CPU "
                              "oracle in the cpu_baseline of the cuda line"}))
            return
        run_backward(args)
        return
    if args.op == "mm_reduce_scatter":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--op mm_reduce_scatter has "
                              "its CPU oracle in the cpu_baseline of the cuda line"}))
            return
        run_mmrs(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
