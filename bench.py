#!/usr/bin/env python3
"""Benchmark of the verify-and-sample step on GB300.

One step = one spec_verify call over one batch (every row of the hot path:
row read, max/log-sum-exp, top-k/top-p threshold, acceptance, scan, residual or
bonus sampling). Metric: verified logit rows/s, rows = B*(2K+1) per step, and
the achieved HBM GB/s of the kernel against the measured copy bandwidth.

Default workload: B=64, K=4, V=151,936 bf16, T=0.6, top_p=0.95, no top-k
(the nucleus serving batch). Inputs are synthetic (seeded Zipf-plus-noise
logits); several input sets rotate so that every step reads HBM (each set is
larger than L2 or the rotation spans more than twice L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference   # the float64 CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
KERNEL_NAME = "keyhist_kernel"     # dominant kernel of sampled bf16 batches
FP32_KERNEL = "fstream_kernel"     # dominant kernel of sampled fp32 batches
CLUSTER_KERNEL = "sv_kernel"       # dominant kernel of small batches
GREEDY_KERNEL = "greedy_kernel"    # dominant kernel of temperature-0 workloads


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rk = int(os.environ.get("RANK", "0"))
    lr = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rk, lr


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# Sources of the translation unit that holds the profiled kernels (keyhist_kernel,
# greedy_kernel, the cluster kernel): a profile's counters stay valid while these
# bytes are unchanged; other translation units do not affect those kernels.
PROFILED_SOURCES = ("speculative_decoding_verification_30_gb300/csrc/spec_verify.cu",
                    "speculative_decoding_verification_30_gb300/csrc/keyhist.cuh",
                    "speculative_decoding_verification_30_gb300/csrc/fstream.cuh",
                    "speculative_decoding_verification_30_gb300/csrc/sv_device.cuh",
                    "speculative_decoding_verification_30_gb300/csrc/launch_cache.h",
                    "include/spec_verify.h")


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in PROFILED_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def dominant_kernel(workload: str) -> str:
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS
    w = WORKLOADS[workload]
    if workload == "greedy":
        return GREEDY_KERNEL
    if w.B * (w.K + 1) < 16:
        return CLUSTER_KERNEL
    return KERNEL_NAME if str(w.dtype).endswith("bfloat16") else FP32_KERNEL


def launches_per_call(workload: str) -> int:
    """Kernels one spec_verify call launches on this workload's 16-byte aligned rows:
    greedy_kernel, then (with draft logits and at least 16 rows) keyhist_kernel for
    bf16 rows or fs_order_kernel and fstream_kernel for fp32 rows, then the cluster
    kernel sv_kernel."""
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS
    w = WORKLOADS[workload]
    if workload == "greedy":
        return 1                                   # no draft logits: greedy_kernel alone
    if w.B * (w.K + 1) < 16:
        return 2
    return 3 if str(w.dtype).endswith("bfloat16") else 4


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", f"{dominant_kernel(workload)}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"source_hash:\s*(\w+)", txt)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != source_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def job_throughput(total_ms: float, steps: int, rows_per_step: int, ws: int, dev):
    """Whole-job throughput of `ws` independent replicas.

    Every rank processes `rows_per_step` rows per step on its own inputs; the job
    time is the slowest rank's timed region (max over ranks), and the value is
    the rows all ranks processed divided by that time. Returns (ms_per_step,
    rows/s)."""
    if ws > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([float(total_ms)], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / steps
    return ms_per_step, rows_per_step * ws * steps / (total_ms / 1e3)


def replica_input_step(rank: int, s: int) -> int:
    """Seed index of input set `s` on `rank`: replicas never share inputs."""
    return 1000 * rank + s


def make_sets(w, rank, dev, greedy):
    """Input sets of workload w resident in HBM (rotated so every step reads HBM),
    with drafted tokens from the library's own draft sampler (not timed)."""
    import torch

    import speculative_decoding_verification_30_gb300 as sv
    from speculative_decoding_verification_30_gb300.workloads import make_batch

    set_bytes = w.bytes_per_step(needed_only=True, greedy=greedy)
    nsets = max(2, -(-3 * L2_BYTES // max(1, set_bytes)))
    nsets = min(nsets, 64)
    sets = []
    for s in range(nsets):
        b = make_batch(w, replica_input_step(rank, s), device=dev)
        T, k, P = b.temperature.to(dev), b.top_k.to(dev), b.top_p.to(dev)
        dtok = sv.spec_sample(b.draft, T, k, P, seed=4242, offset=10_000 + s)
        sets.append((b.target, None if greedy else b.draft, dtok, T, k, P))
    torch.cuda.synchronize()
    return sets, set_bytes


def time_steps(w, sets, steps, warmup, rank, dev, ws=1, stream=None):
    """W untimed warm-up calls, then K timed calls between CUDA events on the
    launching stream (barrier + synchronize on both sides). Returns (total_ms,
    mean per-call ms, clock summary)."""
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_30_gb300 as sv

    B, K = w.B, w.K
    nsets = len(sets)
    wspace = sv.Workspace(B, K, dev)
    out_tok = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    out_n = torch.empty(B, dtype=torch.int32, device=dev)
    stream = stream or torch.cuda.current_stream()

    def step(t):
        tg, dr, dt, T, k, P = sets[t % nsets]
        sv.spec_verify(tg, dr, dt, T, k, P, seed=1234 + rank, offset=t, out_tokens=out_tok,
                       out_n=out_n, workspace=wspace, stream=stream)

    for t in range(warmup):
        step(t)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for t in range(steps):
            starts[t].record(stream)
            step(warmup + t)
            ends[t].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.25)
    if ws > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    per_launch_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    return total_ms, per_launch_ms, clk.summary(), wspace, out_tok, out_n


def other_workloads(args, dev, peak):
    """The other bench-size workloads, measured in the same process: the greedy
    batch (B=256), the mixed fp32 batch (B=512) and the B=1 MTP decode shape."""
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS
    res = {}
    for name, steps in (("greedy", 100), ("mixed", 20), ("mtp_decode", 200)):
        w = WORKLOADS[name]
        greedy = name == "greedy"
        sets, _ = make_sets(w, 0, dev, greedy)
        total_ms, per_ms, clocks, *_ = time_steps(w, sets, steps, 5, 0, dev)
        alg = w.bytes_per_step(needed_only=True, greedy=greedy)
        ach = alg / (per_ms / 1e3) / 1e9
        entry = {"config": {"B": w.B, "K": w.K, "V": w.V, "description": w.description},
                 "ms_per_step": total_ms / steps, "launch_ms": per_ms,
                 "value": w.rows_per_step() / (total_ms / steps / 1e3), "unit": "rows/s",
                 "alg_bytes_per_step": alg, "achieved_GBps": ach, "frac": ach / peak,
                 "kernel": dominant_kernel(name), "gpu_launches_per_step": launches_per_call(name),
                 "clocks": clocks, "steps": steps}
        if name == "greedy":
            entry["bytes_note"] = ("needed bytes (target rows only; greedy reads no draft rows); "
                                   f"the formula B(2K+1)Vs gives {w.bytes_per_step()} B")
        res[name] = entry
        del sets
    return res


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def greedy_from_hidden(dev, steps: int = 20, warmup: int = 3):
    """The greedy batch's shape computed from hidden states (B = 256, K = 3,
    V = 151,936, d = 1,024, bf16): the LM-head GEMM with the argmax epilogue and
    the acceptance kernel (spec_verify_greedy_from_hidden, no logit row written)
    against the GEMM writing fp32 rows followed by spec_verify on them
    (spec_verify_from_hidden). CUDA events around each call; W (311 MB) is larger
    than L2."""
    import torch
    import speculative_decoding_verification_30_gb300 as sv
    from speculative_decoding_verification_30_gb300.workloads import hidden_batch
    B, K, V, d = 256, 3, 151_936, 1024
    h, W = hidden_batch(B, K + 1, d, V, seed=1, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    dtok = torch.randint(0, V, (B, K), generator=g, device=dev, dtype=torch.int32)
    ws = sv.Workspace(B, K, dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    ot, on = torch.empty(B, K + 1, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev)
    ot2, on2 = torch.empty_like(ot), torch.empty_like(on)
    scratch = torch.empty(B * (2 * K + 1) * V, dtype=torch.float32, device=dev)
    T = torch.zeros(B, device=dev)
    kk = torch.zeros(B, dtype=torch.int32, device=dev)
    P = torch.ones(B, device=dev)

    def fused():
        sv.spec_verify_greedy_from_hidden(h, W, dtok, flag=flag, out_tokens=ot, out_n=on, workspace=ws)

    def unfused():
        sv.spec_verify_from_hidden(h, W, None, None, dtok, T, kk, P, logits_scratch=scratch, flag=flag,
                                   out_tokens=ot2, out_n=on2, workspace=ws)

    def timed(fn):
        for _ in range(warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    clk = ClockSampler(dev.index or 0)
    with clk:
        ms_f = timed(fused)
        ms_u = timed(unfused)
    agree = bool(torch.equal(ot, ot2) and torch.equal(on, on2)) and int(flag.item()) == 0
    flops = 2.0 * B * (K + 1) * V * d
    peak, src = measured_bf16_tflops()
    tf = flops / (ms_f / 1e3) / 1e12
    del scratch
    return {"config": {"B": B, "K": K, "V": V, "d": d, "hidden": "bf16 0.5 N(0,1)",
                       "weight": "bf16 0.1 N(0,1)", "drafted": "random ids"},
            "fused_ms": ms_f, "unfused_ms": ms_u, "speedup": ms_u / ms_f,
            "fused_TFLOPs": tf, "roofline": {"bound": "tensor", "achieved": tf, "peak": peak,
                                             "unit": "TFLOP/s", "frac": tf / peak, "peak_source": src},
            "logit_bytes_not_written": B * (K + 1) * V * 4, "fused_equals_unfused": agree,
            "clocks": clk.summary(), "steps": steps}


def bench_gpu(args):
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_30_gb300 as sv
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS

    ws, rank, lrank = dist_env()
    torch.cuda.set_device(lrank)
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", lrank)
    w = WORKLOADS[args.workload]
    if args.batch:
        # a smaller batch of the same workload, for profiler captures
        w = dataclasses.replace(w, B=args.batch)
    B, K, V = w.B, w.K, w.V
    greedy = args.workload == "greedy"
    sv.load()

    sets, set_bytes = make_sets(w, rank, dev, greedy)
    nsets = len(sets)
    stream = torch.cuda.current_stream()
    total_ms, per_launch_ms, clocks, wspace, out_tok, out_n = time_steps(
        w, sets, args.steps, args.warmup, rank, dev, ws, stream)
    rows_per_step = w.rows_per_step()
    ms_per_step, value = job_throughput(total_ms, args.steps, rows_per_step, ws, dev)

    # end to end through the public call with host buffers: every step copies its
    # inputs host->device, verifies, and copies tokens and n back. Two device input
    # sets and a copy stream let step t+1's copy overlap step t's verify (the copy,
    # at the host link's bandwidth, is the longer of the two).
    e2e = None
    if not args.no_e2e:
        tg, dr, dt, T, k, P = sets[0]
        h = [x.cpu().pin_memory() if x is not None else None for x in (tg, dr, dt, T, k, P)]
        dbufs = [[torch.empty_like(x) if x is not None else None for x in (tg, dr, dt, T, k, P)]
                 for _ in range(2)]
        h_tok = [torch.empty(B, K + 1, dtype=torch.int32).pin_memory() for _ in range(2)]
        h_n = [torch.empty(B, dtype=torch.int32).pin_memory() for _ in range(2)]
        outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                 torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in h if x is not None)
        d2h = h_tok[0].numel() * 4 + h_n[0].numel() * 4
        e_steps = max(3, min(args.steps, 20))
        copy_stream = torch.cuda.Stream(device=dev)
        freed = [torch.cuda.Event(), torch.cuda.Event()]    # buffer set j is free again
        for ev in freed:
            ev.record(stream)

        def e2e_step(t):
            j = t % 2
            copy_stream.wait_event(freed[j])
            with torch.cuda.stream(copy_stream):
                for src, dst in zip(h, dbufs[j]):
                    if src is not None:
                        dst.copy_(src, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(copy_stream)
            stream.wait_event(ready)
            b = dbufs[j]
            sv.spec_verify(b[0], b[1], b[2], b[3], b[4], b[5], seed=7, offset=t,
                           out_tokens=outs[j][0], out_n=outs[j][1], workspace=wspace,
                           stream=stream)
            h_tok[j].copy_(outs[j][0], non_blocking=True)
            h_n[j].copy_(outs[j][1], non_blocking=True)
            freed[j].record(stream)

        for t in range(2):
            e2e_step(t)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_event(a)
        for t in range(e_steps):
            e2e_step(t)
        z.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(z) / e_steps
        e2e = {"value": rows_per_step * ws / (e_ms / 1e3), "unit": "rows/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms,
               "pipeline": "two input sets; step t+1's host-to-device copy overlaps step t's verify"}

    peak, peak_src = measured_peak()
    alg_bytes = w.bytes_per_step(needed_only=True, greedy=greedy)
    achieved = alg_bytes / (per_launch_ms / 1e3) / 1e9
    line = {
        "metric": "verified logit rows/s at V=151,936 bf16; achieved HBM GB/s vs GB300 peak",
        "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype.__repr__().endswith("bfloat16") else "f32",
        "data": "synthetic (seeded Zipf-plus-noise logits; drafts from the library's sampler)",
        "config": {"workload": w.name, "B": B, "K": K, "V": V, "description": w.description,
                   "rows_per_step": rows_per_step, "input_sets": nsets,
                   "l2": f"{nsets} rotating input sets of {set_bytes / 1e6:.1f} MB (> 2x L2)",
                   "parallelism": f"replicas x{ws}"},
        "achieved_GBps": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None if args.batch else profiled_traffic(w.name),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "alg_bytes_per_launch": alg_bytes,
                     "launch_ms": per_launch_ms, "kernel": dominant_kernel(w.name),
                     "timing": "CUDA events around each spec_verify call (all kernels of "
                               "the call), so the dominant kernel's own fraction is at "
                               "least this"},
        "gpu_launches": launches_per_call(w.name) * args.steps,
        "e2e": e2e,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_others and args.workload == "nucleus_batch":
        del sets
        torch.cuda.empty_cache()
        line["other_workloads"] = other_workloads(args, dev, peak)
        torch.cuda.empty_cache()
        line["other_workloads"]["greedy_from_hidden"] = greedy_from_hidden(dev)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()


def _oracle_seq(job):
    """One sequence through the oracle (a process-pool task)."""
    from oracle import sampler
    tg, dr, d, T, k, P, step, s = job
    sampler.verify_sequence(tg, dr, d, T, k, P, 1, step, s)
    return 1


def _oracle_jobs(w, step, nb):
    from speculative_decoding_verification_30_gb300.workloads import (draft_tokens_by_rank,
                                                                       make_batch)
    b = make_batch(w, 50_000 + step, B=min(nb, w.B))
    dtok = draft_tokens_by_rank(b.draft, step, w.cid)
    tg = b.target.float().double().numpy()
    dr = b.draft.float().double().numpy()
    return [(tg[s], dr[s], dtok[s].tolist(), float(b.temperature[s]), int(b.top_k[s]),
             float(b.top_p[s]), step, s) for s in range(tg.shape[0])]


def cpu_baseline(w, budget_s: float = 15.0, all_cores: bool = True):
    """The float64 oracle, as it stands, on the host over a bounded sample of the
    workload: single-threaded, and (all_cores) a spawn-started process pool over
    sequences on every host core. value = the all-cores rate when measured."""
    import multiprocessing as mp

    host_cores = os.cpu_count() or 1
    nb = 2 if w.V > 10_000 else w.B
    done_rows, spent, seqs, step = 0, 0.0, 0, 0
    single_budget = budget_s / 2 if all_cores and host_cores > 1 else budget_s
    while spent < single_budget and step < 10_000:
        jobs = _oracle_jobs(w, step, nb)
        t0 = time.perf_counter()
        for j in jobs:
            _oracle_seq(j)
        spent += time.perf_counter() - t0
        seqs += len(jobs)
        done_rows += len(jobs) * (2 * w.K + 1)
        step += 1
    v1 = done_rows / spent
    out = {"value": v1, "unit": "rows/s", "cores": 1, "kind": "oracle", "host_cores": host_cores,
           "value_1core": v1,
           "sample": f"{seqs} sequences of {w.name} (K={w.K}, V={w.V}), {spent:.1f} s "
                     f"single-threaded float64 NumPy"}
    if all_cores and host_cores > 1:
        # enough sequences for every core to stay busy for about half the budget
        per_seq = spent / max(1, seqs)
        n_all = max(host_cores, int(host_cores * (budget_s / 2) / max(per_seq, 1e-6)))
        jobs, st = [], 0
        while len(jobs) < n_all:
            jobs += _oracle_jobs(w, 20_000 + st, max(nb, host_cores))
            st += 1
        jobs = jobs[:n_all]
        with mp.get_context("spawn").Pool(host_cores) as pool:
            pool.map(_oracle_seq, jobs[:host_cores])           # start the workers
            t0 = time.perf_counter()
            pool.map(_oracle_seq, jobs, chunksize=1)
            dt = time.perf_counter() - t0
        va = len(jobs) * (2 * w.K + 1) / dt
        out.update({"value": va, "cores": host_cores, "value_all_cores": va,
                    "sample": out["sample"] + f"; then {len(jobs)} sequences in {dt:.1f} s on a "
                              f"{host_cores}-process pool (one sequence per task)"})
    return out


def bench_reference(args):
    """Reference arm: the CPU oracle, timed as it stands, on bounded samples."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    budget = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(w, budget_s=0.5, all_cores=False)
    vals = [cpu_baseline(w, budget_s=budget) for _ in range(args.steps)]
    value = statistics.mean(v["value"] for v in vals)
    ms_per_step = 1e3 * w.rows_per_step() / value
    line = {
        "impl": "reference",
        "metric": "verified logit rows/s at V=151,936 bf16; achieved HBM GB/s vs GB300 peak",
        "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V,
                   "description": w.description},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": vals[0]["cores"],
                         "host_cores": vals[0]["host_cores"], "kind": "oracle",
                         "value_1core": statistics.mean(v["value_1core"] for v in vals),
                         "value_all_cores": (statistics.mean(v["value_all_cores"] for v in vals)
                                             if "value_all_cores" in vals[0] else None),
                         "sample": vals[0]["sample"]},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="nucleus_batch")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the greedy, mixed and MTP-decode workloads measured after the headline")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size B (profiler captures on a small case)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
