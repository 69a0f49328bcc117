"""Benchmark: exact attention fwd+bwd on GB300, TFLOP/s and % of dense BF16 peak.

One step = the whole path on one batch: fa_fwd_ws (O, lse) then fa_bwd (prep ->
D, main -> dK, dV, dq -> dQ) on the workload B=4 H=16 N=4096 d=128, causal,
bf16 inputs resident in HBM.  FLOPs per step follow the convention
4*B*H*N^2*d for the forward, halved for causal, and 2.5x that for the
backward.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle (the only reference this project
has) on the host cores, on a bounded sample of the same workload per step.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: every
rank runs the full workload, no data-path collective; value = all ranks' FLOPs
divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s at 1 GB300 (bf16) and % of dense BF16 tensor peak"
WORKLOAD = "fwdbwd_4k_d128"
FWD_GATE_WORKLOAD = "fwd_8k_d128_kx3"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def fwd_flops(w, causal=True):
    return 4.0 * w.B * w.H * w.N * w.N * w.d / (2.0 if causal else 1.0)


KERNEL_SOURCES = {"fa_bwd_dkdv_kernel<128>": ("fa_bwd.cu", "ptx.cuh", "fa_internal.cuh"),
                  "fa_bwd_dq_kernel<128>": ("fa_bwd_dq.cu", "ptx.cuh", "fa_internal.cuh"),
                  "fa_fwd_kernel<128>": ("fa_fwd.cu", "ptx.cuh", "fa_internal.cuh"),
                  "fa_fwd_fp8_kernel": ("fa_fp8.cu", "ptx.cuh", "fa_internal.cuh")}


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when no capture exists or the kernel's sources changed since it was taken."""
    import glob
    import hashlib
    srcs = KERNEL_SOURCES.get(kernel)
    if not srcs:
        return None
    h = hashlib.sha256()
    for f in srcs:
        with open(os.path.join(ROOT, "exact_tiled_attention_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    sha = h.hexdigest()
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(path) as fh:
            for line in fh:
                if not line.startswith("bench-traffic:"):
                    continue
                fields = dict(kv.split("=", 1) for kv in line.split()[1:])
                if fields.get("kernel") == kernel and fields.get("source_sha256") == sha:
                    return int(fields["bytes"])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl != "reference" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="fa_clocks_", suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        self.proc = subprocess.Popen(
            [exe, "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
             "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = sorted(r[0] for r in rows)
        reasons = sorted({name for r in rows for name, v in zip(self.REASONS, r[3]) if v == "Active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def oracle_baseline(w, inputs_cpu, target_s=12.0, max_heads=64):
    """fp64 oracle fwd+bwd on whole heads of the workload, all host cores,
    adding heads until about `target_s` seconds of CPU work."""
    import oracle
    from exact_tiled_attention_05_gb300 import workloads as wl
    bits = {n: wl.bf16_bits(t) for n, t in inputs_cpu.items()}
    threads = oracle.default_threads()
    per_head = fwd_flops(w) / w.BH * 3.5  # fwd + 2.5x bwd
    done, spent = 0, 0.0
    while done < max_heads and spent < target_s:
        t0 = time.perf_counter()
        oracle.bwd(bits["q"], bits["k"], bits["v"], bits["do"], w.scale, True, heads=[done],
                   nthreads=threads)
        spent += time.perf_counter() - t0
        done += 1
    return {"value": per_head * done / spent / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of {done} of {w.BH} heads (N={w.N}, d={w.d}, causal), "
                      f"{spent:.1f} s on {threads} host threads"}


def oracle_forward_rates(threads, budget_s=1.0):
    """The fp64 oracle's forward beside the other four workloads: per workload and
    mask, seeded query rows of one head (all rows of the 256-row head), adding rows
    until a call takes about `budget_s` seconds (calls on the 256-row head are
    repeated to fill it); on every host thread and, for the two small workloads,
    on one thread too.  FLOPs are those of the rows evaluated (4·d per visible
    key, so causal rows count only their own keys)."""
    import numpy as np
    import oracle
    from exact_tiled_attention_05_gb300 import workloads as wl
    out = {}
    for name in ("single_head_256", "fwd_2k_d64", "fwd_8k_d128_kx3", "fwd_32k_d128"):
        w = wl.WORKLOADS[name]
        inp = wl.make_inputs(w, B=1, H=1)
        b = {n: wl.bf16_bits(inp[n]) for n in ("q", "k", "v")}
        for causal in w.causal_modes:
            for nt in ((threads, 1) if w.N <= 2048 else (threads,)):
                count = min(16, w.N)
                while True:
                    rows = wl.sampled_rows(w, count=count, BH=1, N=w.N)
                    reps, spent = 0, 0.0
                    while spent < budget_s and (reps == 0 or count == w.N):
                        t0 = time.perf_counter()
                        oracle.fwd_rows(b["q"], b["k"], b["v"], w.scale, causal, rows, nthreads=nt)
                        spent += time.perf_counter() - t0
                        reps += 1
                    if spent >= budget_s / 2 or count == w.N:
                        break
                    count = min(w.N, count * 4)
                keys = (rows[0] + 1) if causal else np.full(rows.shape[1], w.N)
                flops = 4.0 * w.d * float(keys.sum()) * reps
                mode = "causal" if causal else "non-causal"
                out[f"{name} {mode}, {nt} thread{'s' if nt > 1 else ''}"] = {
                    "gflops": flops / spent / 1e9, "rows": int(rows.shape[1]), "calls": reps,
                    "seconds": round(spent, 3)}
    return out


def run_reference(args, world, rank):
    """--impl reference: the oracle on the host cores, same metric and config."""
    from exact_tiled_attention_05_gb300 import workloads as wl
    import oracle
    w = wl.WORKLOADS[WORKLOAD]
    if rank != 0:
        return
    threads = oracle.default_threads()
    # Each step: fwd+bwd of the causal prefix of n positions of one head, with n
    # chosen so the whole run stays within about two minutes.
    full = wl.make_inputs(w, B=1, H=1)
    bits = {nm: wl.bf16_bits(t) for nm, t in full.items()}
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)

    def run_prefix(n):
        sl = {nm: b[:, :n].copy() for nm, b in bits.items()}
        t0 = time.perf_counter()
        oracle.bwd(sl["q"], sl["k"], sl["v"], sl["do"], w.scale, True, nthreads=threads)
        return time.perf_counter() - t0

    n = 128
    t = run_prefix(n)
    while n < w.N and t * 4 < budget:
        n *= 2
        t = run_prefix(n)
    n = min(n, w.N)
    flops = 4.0 * n * n * w.d / 2.0 * 3.5
    for _ in range(args.warmup):
        run_prefix(n)
    times = [run_prefix(n) for _ in range(args.steps)]
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"fp64 oracle fwd+bwd of the first {n} positions (causal) of one head of "
              f"B={w.B} H={w.H} N={w.N} d={w.d} per step, {threads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": f"attention fwd+bwd B={w.B} H={w.H} N={w.N} d={w.d} causal",
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True, "scale": "1/sqrt(d)",
            "inputs": "bf16 iid N(0,1) Q, K, V, dO from a seeded CPU generator",
            "l2": "no flush: Q, K, V, dO alone are 268 MB, larger than the 129 MB L2",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, world, rank, local):
    import torch
    import exact_tiled_attention_05_gb300 as fa
    from exact_tiled_attention_05_gb300 import workloads as wl

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()
    w = wl.WORKLOADS[WORKLOAD]
    B, H, N, d = w.B, w.H, w.N, w.d
    peaks, peak_src = load_peaks()

    cpu_in = wl.make_inputs(w)  # q, k, v, do (bf16, CPU)
    q, k, v, do = (cpu_in[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.alloc_workspace(B, H, N, d, dev)
    fws = torch.empty(fa.fa_fwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    h = stream.cuda_stream
    scale = w.scale
    P = lambda t: t.data_ptr()

    def check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: {fa.status_string(rc)}")

    def step():
        # one step through the public calls: the forward, then the backward
        # (fa_bwd runs prep, dK/dV and dQ)
        check(fa.fa_fwd_ws(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, 1, P(fws), fws.numel(),
                           h), "fa_fwd_ws")
        check(fa.fa_bwd(P(q), P(k), P(v), P(o), P(lse), P(do), P(dq), P(dk), P(dv), B, H, N, d, scale,
                        1, P(ws), ws.numel(), h), "fa_bwd")

    def step_staged(ev):
        # the same step with the backward's three stages called one by one and
        # CUDA events between the four kernels
        ev[0].record(stream)
        check(fa.fa_fwd_ws(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, 1, P(fws), fws.numel(),
                           h), "fa_fwd_ws")
        ev[1].record(stream)
        check(fa.fa_bwd_prep(P(o), P(do), P(lse), B, H, N, d, P(ws), ws.numel(), h), "fa_bwd_prep")
        ev[2].record(stream)
        check(fa.fa_bwd_main(P(q), P(k), P(v), P(lse), P(do), P(dk), P(dv), B, H, N, d, scale, 1,
                             P(ws), ws.numel(), h), "fa_bwd_main")
        ev[3].record(stream)
        check(fa.fa_bwd_dq(P(q), P(k), P(v), P(lse), P(do), P(dq), B, H, N, d, scale, 1, P(ws),
                           ws.numel(), h), "fa_bwd_dq")
        ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check(fa.fa_sync_status(h), "warm-up")

    # ---------------- timed region: K steps on resident inputs ----------------
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    check(fa.fa_sync_status(h), "timed region")
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # ---------------- per-kernel times: the staged step, events between kernels ----------------
    # (each interval includes its kernel's launch gap and, for the stages called
    # on their own, the memset of their work counter)
    n_staged = max(3, min(args.steps, 200))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_staged)]
    torch.cuda.synchronize(dev)
    for i in range(n_staged):
        step_staged(evs[i])
    torch.cuda.synchronize(dev)
    check(fa.fa_sync_status(h), "staged steps")
    per = {name: sum(e[a].elapsed_time(e[b]) for e in evs) / n_staged
           for name, a, b in (("fwd", 0, 1), ("bwd_prep", 1, 2), ("bwd_dkdv", 2, 3),
                              ("bwd_dq", 3, 4))}
    f_fwd = fwd_flops(w)
    f_step = 3.5 * f_fwd
    value = f_step * args.steps * world / (elapsed_ms / 1e3) / 1e12
    ms_step = elapsed_ms / args.steps

    # dominant kernel.  Algorithmic FLOPs per launch: the forward's two MMAs
    # (S, P V) are f_fwd; the dK/dV kernel's four (S, dP, dV, dK) 2 f_fwd; the
    # dQ kernel's dQ = dS K 0.5 f_fwd (its recomputed S and dP are overhead).
    dom = max(per, key=per.get)
    dom_flops = {"fwd": f_fwd, "bwd_dkdv": 2.0 * f_fwd, "bwd_dq": 0.5 * f_fwd}.get(dom)
    achieved = dom_flops / (per[dom] / 1e3) / 1e12 if dom_flops else None
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak, peak_kind = choose_peak(peaks, peak_src, elapsed_ms, clk)
    roofline = {
        "kernel": {"bwd_dkdv": "fa_bwd_dkdv_kernel<128>", "bwd_dq": "fa_bwd_dq_kernel<128>",
                   "fwd": "fa_fwd_kernel<128>"}.get(dom, dom),
        "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
        "frac": achieved / peak if achieved else None,
        "peak_kind": peak_kind,
        "frac_burst": achieved / peak_burst if achieved else None,
        "frac_sustained": achieved / peak_sus if achieved else None,
        "traffic": None,
        "traffic_note": "dram__bytes_read.sum + dram__bytes_write.sum per launch from the committed "
                        "ncu capture under profiles/; null when the kernel changed since",
        "flops_per_launch": dom_flops,
        "ms_per_launch": per[dom],
    }

    # every kernel of the step against its own bound: the three tensor-core kernels
    # in algorithmic TFLOP/s (the dQ kernel also in MMA work: its recomputed S and
    # dP make it 1.5 f_fwd of products), prep in algorithmic GB/s against the
    # measured copy bandwidth
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    prep_bytes = (4 * w.N * w.d + 12 * w.N) * w.B * w.H
    kernels = {}
    for name, flops, mma in (("fwd", f_fwd, f_fwd), ("bwd_dkdv", 2.0 * f_fwd, 2.0 * f_fwd),
                             ("bwd_dq", 0.5 * f_fwd, 1.5 * f_fwd)):
        t = flops / (per[name] / 1e3) / 1e12
        kernels[name] = {"ms": per[name], "tflops": t, "frac": t / peak,
                         "frac_burst": t / peak_burst, "frac_sustained": t / peak_sus,
                         "mma_tflops": mma / (per[name] / 1e3) / 1e12}
    gbs = prep_bytes / (per["bwd_prep"] / 1e3) / 1e9
    kernels["bwd_prep"] = {"ms": per["bwd_prep"], "gbs": gbs, "frac_of_hbm": gbs / hbm}

    kname = roofline["kernel"]
    roofline["traffic"] = profiled_traffic(kname)
    if roofline["traffic"] is not None:
        alg = {"fa_bwd_dkdv_kernel<128>": (12 * w.N * w.d + 8 * w.N) * w.B * w.H,
               "fa_bwd_dq_kernel<128>": (10 * w.N * w.d + 8 * w.N) * w.B * w.H,
               "fa_fwd_kernel<128>": (8 * w.N * w.d + 4 * w.N) * w.B * w.H}.get(kname)
        roofline["algorithmic_bytes"] = alg
        roofline["traffic_over_algorithmic"] = roofline["traffic"] / alg if alg else None

    # ---------------- end to end through the public API, host buffers ----------------
    # Every step copies its inputs in from pinned host memory and its results
    # (O, lse, dQ, dK, dV) back out.  Steps are pipelined over three streams with
    # two sets of device buffers: step k's copy-in and step k-1's copy-out
    # overlap step k-1's / k's compute.
    nbuf = 2
    pin = {n: t.pin_memory() for n, t in cpu_in.items()}
    dev_in = [{n: torch.empty_like(t, device=dev) for n, t in cpu_in.items()} for _ in range(nbuf)]
    dev_out = [{"o": torch.empty_like(o), "lse": torch.empty_like(lse), "dq": torch.empty_like(dq),
                "dk": torch.empty_like(dk), "dv": torch.empty_like(dv)} for _ in range(nbuf)]
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in d_.items()}
                for d_ in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    e2e_steps = max(1, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    cmp_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_run(nsteps):
        for kstep in range(nsteps):
            b = kstep % nbuf
            if kstep >= nbuf:
                s_in.wait_event(cmp_done[b])   # step k-2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                for n in ("q", "k", "v", "do"):
                    dev_in[b][n].copy_(pin[n], non_blocking=True)
                in_done[b].record(s_in)
            s_cmp.wait_event(in_done[b])
            if kstep >= nbuf:
                s_cmp.wait_event(out_done[b])  # step k-2's results have left the device
            x, y = dev_in[b], dev_out[b]
            fa.forward(x["q"], x["k"], x["v"], scale=scale, causal=True, out=y["o"], lse=y["lse"],
                       workspace=fws, stream=s_cmp)
            fa.backward(x["q"], x["k"], x["v"], y["o"], y["lse"], x["do"], scale=scale, causal=True,
                        dq=y["dq"], dk=y["dk"], dv=y["dv"], workspace=ws, stream=s_cmp)
            cmp_done[b].record(s_cmp)
            s_out.wait_event(cmp_done[b])
            with torch.cuda.stream(s_out):
                for n, t in y.items():
                    host_out[b][n].copy_(t, non_blocking=True)
                out_done[b].record(s_out)

    e2e_run(nbuf)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    e2e_run(e2e_steps)
    s_out.wait_event(cmp_done[(e2e_steps - 1) % nbuf])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    check(fa.fa_sync_status(h), "e2e")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": f_step * e2e_steps * world / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "ms_per_step": e2e_ms / e2e_steps,
           "pipeline": "copy-in, compute and copy-out on three streams, two buffer sets",
           "gpu_launches": 4 * e2e_steps}
    del dev_in, dev_out

    # ---------------- sustained: the same step for at least 1.5 s ----------------
    # (the timed region above is exactly --steps steps; this second region shows
    # the rate once the GPU has settled at its power-capped clock)
    sustained = sustained_rate(step, stream, dev, f_step, args.sustained_s, local)

    # ---------------- forward-only workloads ----------------
    # forward gate: N = 8192, d = 128, K x3, causal (inputs 201 MB > L2: no flush)
    wg = wl.WORKLOADS[FWD_GATE_WORKLOAD]
    gin = wl.make_inputs(wg, device=dev)
    fwd_gate = time_forward(fa, wg, gin, True, fws, stream, peak_burst, reps=50, flush=None,
                            hbm_gbs=hbm)
    fwd_gate["gate"] = ">= 60% of dense BF16 peak"
    check(fa.fa_sync_status(h), "forward gate")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > the 129 MB L2
    # B=4 H=16 N=2048 d=64, both masks (inputs 50 MB < L2: L2 flushed before each launch)
    w64 = wl.WORKLOADS["fwd_2k_d64"]
    in64 = wl.make_inputs(w64, device=dev)
    fwd_d64 = {m: time_forward(fa, w64, in64, m == "causal", fws, stream, peak_burst, reps=50,
                               flush=flush, hbm_gbs=hbm) for m in ("non_causal", "causal")}
    # B=1 H=1 N=256 d=64, both masks: a single small launch (latency-bound)
    w1 = wl.WORKLOADS["single_head_256"]
    in1 = wl.make_inputs(w1, device=dev)
    fwd_single = {m: time_forward(fa, w1, in1, m == "causal", fws, stream, peak_burst, reps=50,
                                  flush=flush, hbm_gbs=hbm) for m in ("non_causal", "causal")}
    del flush, in64, in1
    check(fa.fa_sync_status(h), "forward d64")

    # ---------------- FP8 forward (quantize + FP8 attention), same workload ----------------
    fp8 = fp8_forward_timing(fa, wl, wg, gin, dev, stream, peak_burst)
    check(fa.fa_sync_status(h), "fp8 forward")

    del gin

    # ---------------- forward at N = 32768 (the long-context workload), causal ----------------
    wl32 = wl.WORKLOADS["fwd_32k_d128"]
    lin = wl.make_inputs(wl32, device=dev)
    fwd_long = time_forward(fa, wl32, lin, True, fws, stream, peak_burst, reps=10, flush=None,
                            hbm_gbs=hbm)
    fwd_long["gate"] = ">= 60% of dense BF16 peak"
    check(fa.fa_sync_status(h), "forward 32k")
    del lin

    step_bytes = ((8 * N * d + 4 * N) + (12 * N * d + 8 * N) + (10 * N * d + 8 * N)
                  + (4 * N * d + 12 * N)) * B * H
    mhz = clk.get("sm_mhz") if clk else None
    step_line = {"tflops": value / world, "frac": value / world / peak, "peak": peak,
            "peak_kind": peak_kind, "frac_burst": value / world / peak_burst,
            "frac_sustained": value / world / peak_sus,
            "flops_per_step": f_step, "algorithmic_bytes_per_step": step_bytes,
            "timed_region_ms": elapsed_ms,
            "sm_mhz_median": mhz,
            "ms_x_sm_mhz": ms_step * mhz if mhz else None,
            "kcycles_per_step": ms_step * mhz if mhz else None}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": workload_config(w),
        "pct_of_bf16_peak": 100.0 * value / world / peak_burst,
        "peak_bf16_tflops": peak_burst, "peak_source": peak_src,
        "step": step_line, "sustained": sustained,
        "kernel_ms": per, "kernel_ms_steps": n_staged, "kernels": kernels, "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": 4 * args.steps,
        "clocks": clk, "forward_gate": fwd_gate, "forward_gate_long": fwd_long,
        "forward_d64": fwd_d64, "forward_single_head": fwd_single, "fp8_forward": fp8,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, cpu_in)
        line["oracle_forward_rates"] = oracle_forward_rates(line["cpu_baseline"]["cores"])
    if rank == 0:
        print(json.dumps(line), flush=True)


def choose_peak(peaks, peak_src, elapsed_ms, clk):
    """Roofline denominator for kernels timed in the main region: the burst
    BF16 peak (a short matmul loop) unless the timed region lasted seconds and
    its median SM clock sits at or below the clock the sustained peak was
    measured at (power-capped), then the sustained one."""
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    sus_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    mhz = clk.get("sm_mhz") if clk else None
    if elapsed_ms >= 2000.0 and mhz and sus_mhz and mhz <= 1.1 * sus_mhz:
        return sus, (f"bf16_tflops_sustained ({peak_src}): timed region {elapsed_ms / 1e3:.1f} s at "
                     f"a median {mhz:.0f} MHz, near the sustained peak's {sus_mhz:.0f} MHz")
    return burst, (f"bf16_tflops burst ({peak_src}): timed region {elapsed_ms / 1e3:.2f} s at a "
                   f"median {mhz} MHz" + (f" (sustained peak measured at {sus_mhz:.0f} MHz)"
                                          if sus_mhz else ""))


def sustained_rate(step, stream, dev, f_step, seconds, local):
    """The fwd+bwd step repeated for at least `seconds` of device time: TFLOP/s
    and the median SM clock sampled meanwhile."""
    import torch
    if seconds <= 0:
        return None
    probe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    probe[0].record(stream)
    for _ in range(10):
        step()
    probe[1].record(stream)
    torch.cuda.synchronize(dev)
    n = max(10, int(math.ceil(seconds * 1e3 / (probe[0].elapsed_time(probe[1]) / 10))))
    clocks = ClockSampler(local)
    clocks.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = a.elapsed_time(b)
    return {"steps": n, "seconds": ms / 1e3, "ms_per_step": ms / n,
            "tflops": f_step * n / (ms / 1e3) / 1e12, "clocks": clk}


def time_forward(fa, w, inp, causal, fws, stream, peak_burst, reps, flush, hbm_gbs=6779.0):
    """Median CUDA-event time of `reps` forward launches (fa_fwd_ws) on one
    workload; `flush` (a buffer larger than L2) is overwritten before every
    launch, outside the timed events, when the inputs would fit in L2.  Returns
    the line with its own roofline (tensor-bound: algorithmic FLOPs / time
    against the burst BF16 peak; the launches are single and short)."""
    import torch
    o = torch.empty_like(inp["q"])
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=inp["q"].device)
    run = lambda: fa.forward(inp["q"], inp["k"], inp["v"], causal=causal, out=o, lse=lse,
                             workspace=fws)
    for _ in range(3):
        run()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    torch.cuda.synchronize()
    for a_, b_ in ev:
        if flush is not None:
            flush.fill_(1)
        a_.record(stream)
        run()
        b_.record(stream)
    torch.cuda.synchronize()
    ms = sorted(a_.elapsed_time(b_) for a_, b_ in ev)
    med = ms[reps // 2]
    flops = fwd_flops(w, causal)
    tf = flops / (med / 1e3) / 1e12
    alg_bytes = (8 * w.N * w.d + 4 * w.N) * w.B * w.H
    mode = "causal" if causal else "non-causal"
    extra = " K x3" if w.k_scale != 1.0 else ""
    return {"workload": f"fwd B={w.B} H={w.H} N={w.N} d={w.d}{extra} {mode}",
            "ms_median": med, "ms_min": ms[0], "tflops": tf,
            "pct_of_bf16_peak": 100.0 * tf / peak_burst,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_burst, "unit": "TFLOP/s",
                         "frac": tf / peak_burst, "flops_per_launch": flops,
                         "algorithmic_bytes": alg_bytes,
                         "hbm_floor_ms": alg_bytes / (hbm_gbs * 1e9) * 1e3},
            "l2": "flushed before each launch (256 MB write)" if flush is not None
                  else "inputs larger than L2"}


def fp8_forward_timing(fa, wl, wg, gin, dev, stream, peak_bf16, reps=50):
    """FP8 forward on the forward-gate workload: per-tile E4M3 quantization with
    the random-sign Hadamard rotation (fa_fp8_quantize), then the FP8 attention
    (fa_fwd_fp8).  Medians of CUDA-event times over `reps` launches each; the
    FP8 dense peak is the measured bf16 peak times the nominal FP8/BF16 ratio 2."""
    import torch
    B, H, N = wg.B, wg.H, wg.N
    words = wl.sign_bits(wg.seed + 7)
    ws = torch.empty(fa.fp8_workspace_bytes(B, H, N), dtype=torch.uint8, device=dev)
    o = torch.empty_like(gin["q"])
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    quant = lambda: fa.quantize_fp8(gin["q"], gin["k"], gin["v"], signs=words, workspace=ws)
    attn = lambda: fa.forward_fp8_quantized(ws, B, H, N, causal=True, out=o, lse=lse)
    for _ in range(3):
        quant()
        attn()

    def median_ms(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        torch.cuda.synchronize(dev)
        for a_, b_ in ev:
            a_.record(stream)
            fn()
            b_.record(stream)
        torch.cuda.synchronize(dev)
        return sorted(a_.elapsed_time(b_) for a_, b_ in ev)[reps // 2]

    t_attn, t_quant = median_ms(attn), median_ms(quant)
    flops = fwd_flops(wg)
    tf = flops / (t_attn / 1e3) / 1e12
    peak_fp8 = 2.0 * peak_bf16
    alg_bytes = B * H * (3 * N * wg.d + 2 * N * wg.d + 4 * N)  # Q8, K8, V8^T in, O bf16 + lse out
    return {"workload": f"fwd B={B} H={H} N={N} d={wg.d} K x3 causal, Q/K rotated, per-tile E4M3 scales",
            "kernel": "fa_fwd_fp8_kernel", "algorithmic_bytes": alg_bytes,
            "traffic": profiled_traffic("fa_fwd_fp8_kernel"),
            "attention_ms_median": t_attn, "quantize_ms_median": t_quant,
            "tflops": tf, "tflops_incl_quantize": flops / ((t_attn + t_quant) / 1e3) / 1e12,
            "pct_of_fp8_peak": 100.0 * tf / peak_fp8,
            "peak_fp8_tflops": peak_fp8, "peak_fp8_source": "measured bf16 peak x 2 (nominal FP8/BF16 ratio)"}


def run_only(args, local):
    """Untimed launches of one part of the path, for profilers: `fwd` runs the
    forward on the N=8192 d=128 K x3 causal workload, `fwd64` the non-causal
    forward on B=4 H=16 N=2048 d=64, `bwd` the backward (prep, main, dq)
    on the fwd+bwd workload, `fp8` the FP8 quantization (Q/K, V, fold kernels)
    and FP8 attention on the first workload.  W + K launches each."""
    import torch
    import exact_tiled_attention_05_gb300 as fa
    from exact_tiled_attention_05_gb300 import workloads as wl
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()
    if args.only == "fp8":
        w = wl.WORKLOADS[FWD_GATE_WORKLOAD]
        inp = wl.make_inputs(w, device=dev)
        words = wl.sign_bits(w.seed + 7)
        ws = torch.empty(fa.fp8_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
        o = torch.empty_like(inp["q"])
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        for _ in range(args.warmup + args.steps):
            fa.quantize_fp8(inp["q"], inp["k"], inp["v"], signs=words, workspace=ws)
            fa.forward_fp8_quantized(ws, w.B, w.H, w.N, causal=True, out=o, lse=lse)
    elif args.only in ("fwd", "fwd64"):
        w = wl.WORKLOADS[FWD_GATE_WORKLOAD if args.only == "fwd" else "fwd_2k_d64"]
        causal = args.only == "fwd"
        inp = wl.make_inputs(w, device=dev)
        o = torch.empty_like(inp["q"])
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        for _ in range(args.warmup + args.steps):
            fa.forward(inp["q"], inp["k"], inp["v"], causal=causal, out=o, lse=lse)
    else:
        w = wl.WORKLOADS[WORKLOAD]
        inp = wl.make_inputs(w, device=dev)
        o, lse = fa.forward(inp["q"], inp["k"], inp["v"], causal=True)
        ws = fa.alloc_workspace(w.B, w.H, w.N, w.d, dev)
        grads = [torch.empty_like(inp["q"]) for _ in range(3)]
        for _ in range(args.warmup + args.steps):
            fa.backward(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], causal=True,
                        dq=grads[0], dk=grads[1], dv=grads[2], workspace=ws)
    fa.sync_status()
    print(json.dumps({"only": args.only, "launches": args.warmup + args.steps}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-s", type=float, default=1.5,
                    help="seconds of back-to-back steps for the 'sustained' rate (0: skip)")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for the whole run")
    ap.add_argument("--only", choices=("fwd", "fwd64", "bwd", "fp8"), default=None,
                    help="untimed launches of one part of the path (for profilers)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference" and not args.only:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    try:
        if args.only:
            run_only(args, local)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
