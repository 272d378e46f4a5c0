"""Benchmark of the NF4 + double-quantized LoRA linear layer on one B300.

One step = forward + backward of all seven NF4-LoRA projections of a
Llama-3.1-8B-shaped decoder layer (q, k, v, o, gate, up, down; r = 16,
alpha = 32, M = 2048 tokens), inputs resident in HBM. The line also carries
the standalone codec measurement (14336 x 4096 quantize once + dequantize
x100), the roofline of the dominant kernel, an end-to-end figure through the
C ABI with host buffers, and the CPU oracle timed on a bounded token sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own M tokens (weak scaling, data
parallel) and the adapter gradients are all-reduced over NCCL each step.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_lora_double_b300 import dp, synth  # noqa: E402

WORKLOAD = 1          # Llama-3.1-8B-shaped layer, M = 2048, r = 16
CODEC_WORKLOAD = 2    # 14336 x 4096 codec
CPU_SAMPLE_TOKENS = 96
METRIC = "QLoRA linear fwd+bwd TFLOP/s and % bf16 peak; NF4 dequant GB/s and % HBM"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


def sources_sha256():
    """Hash of the library sources (kernels and ABI header)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "bit_quantized_lora_double_b300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "qlora.h"))
    for f in files:
        if os.path.isfile(f):
            h.update(os.path.basename(f).encode())
            h.update(open(f, "rb").read())
    return h.hexdigest()


def measured_traffic(kind):
    """DRAM bytes per launch of a kernel kind from the committed ncu summary,
    or None when the sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("sources_sha256") != sources_sha256():
        return None
    return d.get("per_launch_bytes", {}).get(kind)


def step_flops(M, projections, r):
    return sum(4 * M * n * k + 6 * M * r * (n + k) for _, n, k in projections)


def fwd_gemm_flops(M, n, k, r):
    # one forward main-kernel launch: X W'^T plus the LoRA up-projection
    return 2 * M * n * k + 2 * M * n * r


def dx_gemm_flops(M, n, k, r):
    return 2 * M * n * k + 2 * M * k * r


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.f:
            return None
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(M_tokens, projections, r, scale):
    """The CPU oracle, as it stands, on a bounded token sample of the step."""
    from oracle import oracle
    tot_t, tot_f = 0.0, 0
    for p, (name, n, k) in enumerate(projections):
        X, W, A, B, dY, s = synth.layer_inputs(WORKLOAD, p, M=M_tokens)
        qw = oracle.nf4_quantize(W)
        Wdq = oracle.nf4_dequantize(qw)
        t = time.perf_counter()
        oracle.linear_fwd(X, Wdq, A, B, s)
        oracle.linear_bwd(dY, X, Wdq, A, B, s)
        tot_t += time.perf_counter() - t
        tot_f += 4 * M_tokens * n * k + 6 * M_tokens * r * (n + k)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OMP_NUM_THREADS", cores))
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{M_tokens} tokens of each of the 7 projections, forward + backward (fp64 C loops, "
                      f"OpenMP); {tot_t:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores, per step a bounded
    sample (one token of one projection, round robin)."""
    if rank != 0:
        return
    from oracle import oracle
    w = synth.WORKLOADS[WORKLOAD]
    projs, r = w["projections"], w["r"]
    prep = []
    for p in range(len(projs)):
        X, W, A, B, dY, s = synth.layer_inputs(WORKLOAD, p, M=1)
        qw = oracle.nf4_quantize(W)
        prep.append((X, oracle.nf4_dequantize(qw), A, B, dY, s, projs[p]))

    def one(i):
        X, Wdq, A, B, dY, s, (_, n, k) = prep[i % len(prep)]
        t = time.perf_counter()
        oracle.linear_fwd(X, Wdq, A, B, s)
        oracle.linear_bwd(dY, X, Wdq, A, B, s)
        return time.perf_counter() - t, 4 * n * k + 6 * r * (n + k)

    for i in range(args.warmup):
        one(i)
    tt, ff = 0.0, 0
    for i in range(args.steps):
        t, f = one(args.warmup + i)
        tt += t
        ff += f
    v = ff / tt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "M": w["M"], "r": r, "sample": "1 token of one projection per step"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "1 token of one projection (round robin over q,k,v,o,gate,up,down) per step"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def device_projection(qlora, torch, dev, gen, n, k, M, r, w_std, b_std, copies=1):
    """Seeded device-side inputs of one projection (torch Philox generator,
    the same distributions as the parity inputs): the NF4 weight (and
    `copies` - 1 extra copies of it), X, dY ~ N(0, 1), A ~ N(0, 1/K),
    B ~ N(0, b_std); output buffers and one workspace."""
    bf = torch.bfloat16

    def normal(shape, std):
        return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * std).to(bf)

    W = normal((n, k), w_std)
    w = qlora.alloc_nf4_weight(n, k, dev)
    qlora.qlora_nf4_quantize(W, w, qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k), dev))
    del W
    ws_ = [w]
    for _ in range(copies - 1):
        x = qlora.alloc_nf4_weight(n, k, dev)
        x.codes.copy_(w.codes); x.absmax_q.copy_(w.absmax_q)
        x.absmax_scale.copy_(w.absmax_scale); x.absmax_mean.copy_(w.absmax_mean)
        ws_.append(x)
    d = dict(n=n, k=k, w=ws_, X=normal((M, k), 1.0), dY=normal((M, n), 1.0), A=normal((r, k), 1.0 / k),
             B=normal((n, r), b_std), Y=torch.empty((M, n), dtype=bf, device=dev),
             U=torch.empty((M, r), dtype=bf, device=dev), dX=torch.empty((M, k), dtype=bf, device=dev),
             dA=torch.empty((r, k), dtype=torch.float32, device=dev),
             dB=torch.empty((n, r), dtype=torch.float32, device=dev))
    d["ws"] = qlora.workspace(max(qlora.qlora_linear_fwd_workspace(M, w, r),
                                  qlora.qlora_linear_bwd_workspace(M, w, r)), dev)
    return d


def graph_time(torch, fn, steps, warmup):
    """ms per call of fn, replayed as one CUDA graph per call after warm-up."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def bench_llama70b(qlora, torch, dev, pk, steps):
    """The Llama-70B-shaped projections at M = 4096, r = 64: forward +
    backward of all seven, TFLOP/s."""
    wl = synth.WORKLOADS[3]
    M, r, scale = wl["M"], wl["r"], wl["scale"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(synth.seed_for(3, "X"))
    P = [device_projection(qlora, torch, dev, gen, n, k, M, r, wl["w_std"], wl["b_std"])
         for _, n, k in wl["projections"]]

    def step():
        for d in P:
            qlora.qlora_linear_fwd(d["X"], M, d["w"][0], d["A"], d["B"], r, scale, d["Y"], d["U"], d["ws"])
        for d in reversed(P):
            qlora.qlora_linear_bwd(d["dY"], d["X"], d["U"], M, d["w"][0], d["A"], d["B"], r, scale, d["dX"],
                                   d["dA"], d["dB"], d["ws"])

    ms = graph_time(torch, step, steps, 2)
    flops = step_flops(M, wl["projections"], r)
    out = {"workload": wl["name"] + ": q,k,v,o,gate,up,down NF4+DQ, LoRA r=64 alpha=16", "M": M, "r": r,
           "ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "pct_bf16_peak": flops / (ms * 1e-3) / 1e12 / pk["bf16"],
           "pct_bf16_peak_sustained": flops / (ms * 1e-3) / 1e12 / pk["bf16_sus"]}
    del P
    torch.cuda.empty_cache()
    return out


def bench_sweep(qlora, torch, dev, pk):
    """Token-count sweep on the gate projection 4096 -> 14336 (r = 16): the
    forward at every M, the backward for M >= 128. For M <= 16 the forward
    reads six rotating copies of the packed weight (more than L2 holds) and
    is reported as GB/s against the HBM roofline."""
    wl = synth.WORKLOADS[4]
    _, n, k = wl["projections"][0]
    r, scale = wl["r"], wl["scale"]
    rows = []
    for M in wl["M_sweep"]:
        gen = torch.Generator(device=dev)
        gen.manual_seed(synth.seed_for(4, "X") + M)
        copies = 6 if M <= 16 else 1
        d = device_projection(qlora, torch, dev, gen, n, k, M, r, wl["w_std"], wl["b_std"], copies)
        it = [0]

        def fwd():
            w = d["w"][it[0] % copies]
            it[0] += 1
            qlora.qlora_linear_fwd(d["X"], M, w, d["A"], d["B"], r, scale, d["Y"], d["U"], d["ws"])

        reps = max(3, min(200, int(2e11 / max(1, M * n * k * 2))))
        if copies > 1:
            # eager launches (the rotation over weight copies is host-side)
            for _ in range(5):
                fwd()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fwd()
            b.record()
            torch.cuda.synchronize()
            f_ms = a.elapsed_time(b) / reps
        else:
            f_ms = graph_time(torch, fwd, reps, 3)
        f_fl = 2 * M * n * k + 2 * M * r * (n + k)
        row = {"M": M, "fwd_ms": f_ms, "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12}
        if M <= 16:
            wbytes = n * k // 2 + n * k // 64 + 4 * ((n * k // 64 + 255) // 256) + 4
            byts = wbytes + 2 * (M * k + M * n + r * k + n * r)
            gbs = byts / (f_ms * 1e-3) / 1e9
            row.update({"fwd_gbs": gbs, "fwd_pct_hbm": gbs / pk["hbm"], "fwd_bytes": byts,
                        "l2": "6 rotating weight copies (> L2)"})
        if M >= 128:
            def bwd():
                qlora.qlora_linear_bwd(d["dY"], d["X"], d["U"], M, d["w"][0], d["A"], d["B"], r, scale, d["dX"],
                                       d["dA"], d["dB"], d["ws"])
            b_ms = graph_time(torch, bwd, reps, 3)
            b_fl = 2 * M * n * k + 4 * M * r * (n + k)
            row.update({"bwd_ms": b_ms, "bwd_tflops": b_fl / (b_ms * 1e-3) / 1e12,
                        "fwd_bwd_tflops": (4 * M * n * k + 6 * M * r * (n + k)) / ((f_ms + b_ms) * 1e-3) / 1e12})
        rows.append(row)
        del d
        torch.cuda.empty_cache()
    return {"workload": wl["name"] + ": gate 4096->14336 NF4+DQ, LoRA r=16 alpha=32", "rows": rows}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--prof-steps", type=int, default=20)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the 70B-shaped layer and the M sweep")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist
    from bit_quantized_lora_double_b300 import qlora

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    pk = peaks()

    wl = synth.WORKLOADS[WORKLOAD]
    projs, M, r = wl["projections"], wl["M"], wl["r"]

    def dev_bf16(h):
        return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)

    # ---- setup: quantize the seven weights on the GPU, inputs resident -----
    P = []
    for p, (name, n, k) in enumerate(projs):
        X, W, A, B, dY, s = synth.layer_inputs(WORKLOAD, p)
        w = qlora.alloc_nf4_weight(n, k, dev)
        wsq = qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k), dev)
        qlora.qlora_nf4_quantize(dev_bf16(W), w, wsq)
        del wsq
        d = dict(name=name, n=n, k=k, s=s, w=w, X=dev_bf16(X), A=dev_bf16(A), B=dev_bf16(B), dY=dev_bf16(dY),
                 hX=torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory(),
                 hdY=torch.from_numpy(dY.view(np.int16)).view(torch.bfloat16).pin_memory(),
                 Y=torch.empty((M, n), dtype=torch.bfloat16, device=dev),
                 U=torch.empty((M, r), dtype=torch.bfloat16, device=dev),
                 dX=torch.empty((M, k), dtype=torch.bfloat16, device=dev),
                 dA=torch.empty((r, k), dtype=torch.float32, device=dev),
                 dB=torch.empty((n, r), dtype=torch.float32, device=dev))
        d["ws"] = qlora.workspace(max(qlora.qlora_linear_fwd_workspace(M, w, r),
                                      qlora.qlora_linear_bwd_workspace(M, w, r)), dev)
        P.append(d)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        for d in P:
            qlora.qlora_linear_fwd(d["X"], M, d["w"], d["A"], d["B"], r, d["s"], d["Y"], d["U"], d["ws"])
        for d in reversed(P):
            qlora.qlora_linear_bwd(d["dY"], d["X"], d["U"], M, d["w"], d["A"], d["B"], r, d["s"], d["dX"], d["dA"],
                                   d["dB"], d["ws"])
            if world > 1:
                dp.allreduce_adapter_grads([d["dA"], d["dB"]])

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    qlora.qlora_check_device_status(stream)
    barrier()

    # The timed region replays one CUDA graph of the step (captured after the
    # warm-up; the library's calls allocate and synchronize nothing, so they
    # capture as they are), or launches the step eagerly with --no-graph.
    graph = None
    if not args.no_graph and world == 1:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        barrier()
        qlora.qlora_check_device_status(stream)
    run_step = graph.replay if graph is not None else step

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        ev0.record()
        for _ in range(args.steps):
            run_step()
        ev1.record()
        barrier()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    qlora.qlora_check_device_status(stream)
    clocks = clk.summary()

    flops = step_flops(M, projs, r)
    ms_step = ms / args.steps
    value = world * flops / (ms_step * 1e-3) / 1e12

    # Per-kernel device times: the same step launched eagerly with the
    # library's profiling hooks (a CUDA event pair around every launch, on the
    # launch stream), right after the timed region.
    prof_steps = max(1, min(args.steps, args.prof_steps))
    qlora.qlora_profile_start()
    barrier()
    for _ in range(prof_steps):
        step()
    barrier()
    prof_ms, prof_n, _ = qlora.qlora_profile_stop()
    launches = sum(prof_n.values()) // prof_steps * args.steps

    # dominant kernel of the step and its roofline: per kind, the summed
    # device time of its launches in the timed region against the algorithmic
    # flops of those launches (a kind's split-reduction launches count with it)
    kinds = {k: v for k, v in prof_ms.items() if prof_n[k] > 0}
    dom = max(kinds, key=kinds.get)
    gemm_flops = {"fwd_gemm": sum(fwd_gemm_flops(M, n, k, r) for _, n, k in projs),
                  "fwd_simt": sum(fwd_gemm_flops(M, n, k, r) for _, n, k in projs),
                  "dx_gemm": sum(dx_gemm_flops(M, n, k, r) for _, n, k in projs),
                  "dx_simt": sum(dx_gemm_flops(M, n, k, r) for _, n, k in projs)}
    roof = None
    if dom in gemm_flops:
        ms_kind = prof_ms[dom] / prof_steps
        ach = gemm_flops[dom] / (ms_kind * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_sus"], "traffic": measured_traffic(dom),
                "traffic_note": "DRAM read+write bytes per launch (average over the step's launches) from "
                                "profiles/roofline_traffic.json",
                "peak_note": f"bf16 dense sustained ({pk['src']}); a kernel timed inside a long step",
                "flops_per_launch": gemm_flops[dom] / len(projs),
                "launches_per_step": prof_n[dom] / prof_steps, "ms_per_step": ms_kind,
                "timing": f"CUDA events around each launch, {prof_steps} eager profiled steps after the timed region"}

    # ---- end to end through the C ABI with host buffers ----------------------
    hY = {d["name"]: torch.empty(d["Y"].shape, dtype=torch.bfloat16, pin_memory=True) for d in P}
    hdX = {d["name"]: torch.empty(d["dX"].shape, dtype=torch.bfloat16, pin_memory=True) for d in P}
    hdA = {d["name"]: torch.empty(d["dA"].shape, dtype=torch.float32, pin_memory=True) for d in P}
    hdB = {d["name"]: torch.empty(d["dB"].shape, dtype=torch.float32, pin_memory=True) for d in P}
    h2d = sum(d["hX"].numel() * 2 + d["hdY"].numel() * 2 for d in P)
    d2h = sum(d["Y"].numel() * 2 + d["dX"].numel() * 2 + d["dA"].numel() * 4 + d["dB"].numel() * 4 for d in P)

    # Host copies run on two copy streams beside the compute stream: the inputs
    # of projection p+1 travel while projection p computes, and each result
    # goes back as soon as its kernel is done.
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    comp = torch.cuda.current_stream()

    def e2e_step():
        for d in P:
            with torch.cuda.stream(s_h2d):
                d["X"].copy_(d["hX"], non_blocking=True)
                d["ev_x"] = torch.cuda.Event()
                d["ev_x"].record(s_h2d)
            with torch.cuda.stream(s_h2d):
                d["dY"].copy_(d["hdY"], non_blocking=True)
                d["ev_dy"] = torch.cuda.Event()
                d["ev_dy"].record(s_h2d)
        for d in P:
            comp.wait_event(d["ev_x"])
            qlora.qlora_linear_fwd(d["X"], M, d["w"], d["A"], d["B"], r, d["s"], d["Y"], d["U"], d["ws"])
            ev = torch.cuda.Event()
            ev.record(comp)
            s_d2h.wait_event(ev)
            with torch.cuda.stream(s_d2h):
                hY[d["name"]].copy_(d["Y"], non_blocking=True)
        for d in reversed(P):
            comp.wait_event(d["ev_dy"])
            qlora.qlora_linear_bwd(d["dY"], d["X"], d["U"], M, d["w"], d["A"], d["B"], r, d["s"], d["dX"], d["dA"],
                                   d["dB"], d["ws"])
            if world > 1:
                dp.allreduce_adapter_grads([d["dA"], d["dB"]])
            ev = torch.cuda.Event()
            ev.record(comp)
            s_d2h.wait_event(ev)
            with torch.cuda.stream(s_d2h):
                hdX[d["name"]].copy_(d["dX"], non_blocking=True)
                hdA[d["name"]].copy_(d["dA"], non_blocking=True)
                hdB[d["name"]].copy_(d["dB"], non_blocking=True)
        # the step ends when every result is on the host
        ev = torch.cuda.Event()
        ev.record(s_d2h)
        comp.wait_event(ev)

    e2e_step()
    barrier()
    ev0.record(comp)
    for _ in range(args.e2e_steps):
        e2e_step()
    ev1.record(comp)
    barrier()
    e2e_ms = ev0.elapsed_time(ev1) / args.e2e_steps
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "note": "pinned host buffers; H2D of all inputs and D2H of Y, dX, dA, dB on two copy streams "
                   "overlapping the compute stream"}

    # ---- codec: 14336 x 4096 quantize once + dequantize x100 -----------------
    _, cn, ck = synth.WORKLOADS[CODEC_WORKLOAD]["projections"][0]
    Wc = dev_bf16(synth.gaussian_bf16((cn, ck), 0.02, synth.seed_for(CODEC_WORKLOAD, "W")))
    wc = qlora.alloc_nf4_weight(cn, ck, dev)
    wsc = qlora.workspace(qlora.qlora_nf4_quantize_workspace(cn, ck), dev)
    outc = torch.empty((cn, ck), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        qlora.qlora_nf4_quantize(Wc, wc, wsc)
        qlora.qlora_nf4_dequantize(wc, outc)
    barrier()
    ev0.record(stream)
    qlora.qlora_nf4_quantize(Wc, wc, wsc)
    ev1.record(stream)
    barrier()
    q_ms = ev0.elapsed_time(ev1)
    # rotate over copies of the packed weight larger than L2 in total, so the
    # dequantize reads come from HBM
    ncopy = 6
    wcs = [wc] + [qlora.alloc_nf4_weight(cn, ck, dev) for _ in range(ncopy - 1)]
    for x in wcs[1:]:
        x.codes.copy_(wc.codes); x.absmax_q.copy_(wc.absmax_q)
        x.absmax_scale.copy_(wc.absmax_scale); x.absmax_mean.copy_(wc.absmax_mean)
    outs = [outc] + [torch.empty_like(outc) for _ in range(1)]
    qlora.qlora_profile_start()
    barrier()
    ev0.record(stream)
    for i in range(100):
        qlora.qlora_nf4_dequantize(wcs[i % ncopy], outs[i % 2])
    ev1.record(stream)
    barrier()
    dq_prof_ms, dq_prof_n, _ = qlora.qlora_profile_stop()
    dq_ms = ev0.elapsed_time(ev1) / 100
    dq_kernel_ms = dq_prof_ms["dequant"] / max(1, dq_prof_n["dequant"])
    nel = cn * ck
    dq_bytes = nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4 + 2 * nel
    q_bytes = 2 * nel + nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4
    dq_gbs = dq_bytes / (dq_kernel_ms * 1e-3) / 1e9
    codec = {"workload": "nf4 codec 14336x4096 bf16 N(0,0.02)",
             "dequant": {"value": dq_gbs, "unit": "GB/s", "pct_hbm": dq_gbs / pk["hbm"],
                         "bytes_per_pass": dq_bytes, "ms_per_pass": dq_kernel_ms, "ms_per_call": dq_ms,
                         "l2": f"{ncopy} rotating copies of the packed weight (> L2)",
                         "roofline": {"bound": "hbm", "achieved": dq_gbs, "peak": pk["hbm"], "unit": "GB/s",
                                      "frac": dq_gbs / pk["hbm"], "traffic": measured_traffic("dequant"),
                                      "peak_note": f"HBM copy, {pk['src']}"}},
             "quantize": {"value": q_bytes / (q_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": q_ms,
                          "bytes": q_bytes}}

    extra = {}
    if rank == 0 and world == 1 and not args.no_extra:
        extra["llama70b_layer"] = bench_llama70b(qlora, torch, dev, pk, 5)
        extra["gate_sweep"] = bench_sweep(qlora, torch, dev, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(CPU_SAMPLE_TOKENS, projs, r, wl["scale"])

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "pct_bf16_peak": value / world / pk["bf16"], "pct_bf16_peak_sustained": value / world / pk["bf16_sus"],
            "config": {"workload": wl["name"] + ": q,k,v,o,gate,up,down NF4+DQ, LoRA r=16 alpha=32",
                       "M": M, "r": r, "projections": [[n_, k_] for _, n_, k_ in projs],
                       "flops_per_step": flops, "parallelism": f"dp{world}",
                       "l2": "inputs larger than L2 (about 0.5 GB touched per step)"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "kernels_ms_per_step": {k: v / prof_steps for k, v in prof_ms.items() if prof_n[k]},
            "kernels_launches_per_step": {k: v // prof_steps for k, v in prof_n.items() if v},
            "timed_region": "CUDA graph of one step replayed" if graph is not None else "eager launches",
            "clocks": clocks,
            "codec": codec,
            **extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
