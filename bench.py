"""Benchmark of the NF4 + double-quantized LoRA linear layer on one B300.

One step = forward + backward of all seven NF4-LoRA projections of a
Llama-70B-shaped decoder layer (q, k, v, o, gate, up, down with d_model 8192,
KV width 1024, FFN 28672; LoRA r = 64, alpha = 16; M = 4096 tokens), inputs
resident in HBM, run as the layer runs them: q/k/v on one input and gate/up
on one input, each group as one grouped call (o and down alone), so the
backward returns one input gradient per group. The same step as seven
single-layer calls is timed beside it ("ungrouped"). The same JSON line
carries: the roofline of the step's
dominant kernel kind; an end-to-end figure through the C ABI with host buffers;
the Llama-3.1-8B-shaped layer (M = 2048, r = 16) and the single 1024 x 1024
layer (M = 256, r = 8); the standalone codec (14336 x 4096 quantize once +
dequantize x100); the token sweep on the gate projection; and the CPU oracle
timed on bounded samples.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Every input follows the seeded numpy recipe of synth.py, the same bytes the
parity tests give the oracle. Under torchrun (N > 1) every rank runs its own
M tokens (weak scaling, data parallel) and the adapter gradients are
all-reduced over NCCL each step.
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

WORKLOAD = 3          # Llama-70B-shaped projections, M = 4096, r = 64
LAYER8B = 1           # Llama-3.1-8B-shaped layer, M = 2048, r = 16
SINGLE = 0            # single 1024 x 1024 layer, M = 256, r = 8
CODEC_WORKLOAD = 2    # 14336 x 4096 codec
SWEEP = 4             # gate 4096 -> 14336 token sweep
CPU_SAMPLE_TOKENS = 24
# projections of a decoder layer that read the same input
LAYER_GROUPS = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
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


# algorithmic flops per kernel kind and projection (the LoRA terms that run
# inside the fused GEMMs count with them; U, V, dA, dB are the side path)
KIND_FLOPS = {
    "fwd_gemm": lambda M, n, k, r: 2 * M * n * k + 2 * M * n * r,
    "fwd_simt": lambda M, n, k, r: 2 * M * n * k + 2 * M * n * r,
    "dx_gemm": lambda M, n, k, r: 2 * M * n * k + 2 * M * k * r,
    "dx_simt": lambda M, n, k, r: 2 * M * n * k + 2 * M * k * r,
}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons; `summary` keeps
    the samples taken between mark_start() and mark_end()."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.f = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            # wait for the first sample so the sampler covers the region
            t_end = time.time() + 5
            while time.time() < t_end and os.path.getsize(self.f.name) == 0:
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(2 * self.interval / 1000)

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
        import datetime
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                rows.append((ts, parts[1:]))
        os.unlink(self.f.name)
        inside = [p for ts, p in rows if self.t0 is not None and self.t0 - 0.05 <= ts <= (self.t1 or ts) + 0.05]
        use = inside if inside else [p for _, p in rows]
        if not use:
            return None
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "interval_ms": self.interval}


def workload_name(wl):
    """The headline workload's name, the same on both arms."""
    return (wl["name"] + ": q,k,v,o,gate,up,down NF4+DQ, LoRA r=%d alpha=%g; groups q/k/v, o, gate/up, down"
            % (wl["r"], wl["alpha"]))


def groups_of(P):
    """Index lists of the projections by LAYER_GROUPS (others alone)."""
    names = [d["name"] for d in P]
    out, used = [], set()
    for gr in LAYER_GROUPS:
        idx = [names.index(n) for n in gr if n in names]
        if idx:
            out.append(idx)
            used.update(idx)
    out += [[i] for i in range(len(P)) if i not in used]
    return out


def load_layer(qlora, torch, dev, wl_id, pinned=False):
    """Seeded inputs of every projection of a workload (synth recipe, numpy),
    copied to the device; weights quantized on the GPU; outputs and one
    workspace per projection; pinned host copies of X and dY for the
    end-to-end leg when asked. Projections of one group read the first
    member's X. Returns the workload, the projections and the groups (their
    shared input, stacked U, input gradient and workspace)."""
    wl = synth.WORKLOADS[wl_id]
    M, r = wl["M"], wl["r"]
    P = []
    for p, (name, n, k) in enumerate(wl["projections"]):
        X, W, A, B, dY, s = synth.layer_inputs(wl_id, p)
        dv = lambda h: torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
        w = qlora.alloc_nf4_weight(n, k, dev)
        Wd = dv(W)
        del W
        wsq = qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k), dev)
        qlora.qlora_nf4_quantize(Wd, w, wsq)
        torch.cuda.synchronize()
        del Wd, wsq
        d = dict(name=name, n=n, k=k, s=s, w=w, X=dv(X), A=dv(A), B=dv(B), dY=dv(dY),
                 Y=torch.empty((M, n), dtype=torch.bfloat16, device=dev),
                 U=torch.empty((M, r), dtype=torch.bfloat16, device=dev),
                 dX=torch.empty((M, k), dtype=torch.bfloat16, device=dev),
                 dA=torch.empty((r, k), dtype=torch.float32, device=dev),
                 dB=torch.empty((n, r), dtype=torch.float32, device=dev))
        if pinned:
            d["hX"] = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory()
            d["hdY"] = torch.from_numpy(dY.view(np.int16)).view(torch.bfloat16).pin_memory()
        d["ws"] = qlora.workspace(max(qlora.qlora_linear_fwd_workspace(M, w, r),
                                      qlora.qlora_linear_bwd_workspace(M, w, r)), dev)
        P.append(d)
    G = []
    for idx in groups_of(P):
        first = P[idx[0]]
        for i in idx[1:]:
            P[i]["X"] = first["X"]
            if pinned:
                P[i]["hX"] = first["hX"]
        mem = [P[i] for i in idx]
        ws_, As, Bs = [d["w"] for d in mem], [d["A"] for d in mem], [d["B"] for d in mem]
        G.append(dict(idx=idx, name="/".join(d["name"] for d in mem), X=first["X"], s=first["s"], k=first["k"],
                      w=ws_, A=As, B=Bs, Y=[d["Y"] for d in mem], dY=[d["dY"] for d in mem],
                      dA=[d["dA"] for d in mem], dB=[d["dB"] for d in mem],
                      U=torch.empty((M, len(idx) * r), dtype=torch.bfloat16, device=dev),
                      dX=torch.empty((M, first["k"]), dtype=torch.bfloat16, device=dev),
                      ws=qlora.workspace(max(qlora.qlora_group_fwd_workspace(M, ws_, As, Bs, r),
                                             qlora.qlora_group_bwd_workspace(M, ws_, As, Bs, r)), dev)))
    torch.cuda.synchronize()
    return wl, P, G


def make_group_step(qlora, G, M, r, world):
    """The layer step through the grouped calls."""
    def step():
        for g in G:
            qlora.qlora_group_fwd(g["X"], M, g["w"], g["A"], g["B"], r, g["s"], g["Y"], g["U"], g["ws"])
        for g in reversed(G):
            qlora.qlora_group_bwd(g["X"], g["U"], M, g["w"], g["A"], g["B"], r, g["s"], g["dY"], g["dX"], g["dA"],
                                  g["dB"], g["ws"])
            if world > 1:
                dp.allreduce_adapter_grads(g["dA"] + g["dB"])
    return step


def make_step(qlora, P, M, r, world):
    """The layer step as one single-layer call per projection."""
    def step():
        for d in P:
            qlora.qlora_linear_fwd(d["X"], M, d["w"], d["A"], d["B"], r, d["s"], d["Y"], d["U"], d["ws"])
        for d in reversed(P):
            qlora.qlora_linear_bwd(d["dY"], d["X"], d["U"], M, d["w"], d["A"], d["B"], r, d["s"], d["dX"], d["dA"],
                                   d["dB"], d["ws"])
            if world > 1:
                dp.allreduce_adapter_grads([d["dA"], d["dB"]])
    return step


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    return g


def graph_time(torch, fn, steps, warmup):
    """ms per call of fn, replayed as one CUDA graph per call after warm-up."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = capture(torch, fn)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def profile_kinds(qlora, torch, step, n):
    """Per kernel kind: summed device ms per step and launches per step, from
    CUDA events the library records around each launch on its launch stream
    during n eager steps."""
    torch.cuda.synchronize()
    qlora.qlora_profile_start()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    ms, cnt, _ = qlora.qlora_profile_stop()
    return ({k: v / n for k, v in ms.items() if cnt[k]}, {k: v // n for k, v in cnt.items() if v})


def roofline_of(kind_ms, kind_n, graph_ms, M, projections, r, pk, clocks):
    """Roofline of the dominant kernel kind. Its per-launch device times come
    from the eager profiled steps; they are scaled by (graph step time / sum of
    the kinds' eager times) so that the kinds add up to the timed step, which
    charges any idle time of the graph step to the kernels (a lower bound on
    the rate)."""
    dom = max(kind_ms, key=kind_ms.get)
    if dom not in KIND_FLOPS:
        return None
    scale = graph_ms / sum(kind_ms.values())
    ms_kind = kind_ms[dom] * scale
    fl = sum(KIND_FLOPS[dom](M, n, k, r) for _, n, k in projections)
    ach = fl / (ms_kind * 1e-3) / 1e12
    capped = clocks is not None and "sw_power_cap" in clocks.get("reasons", [])
    return {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": ach / pk["bf16"], "frac_of_sustained_peak": ach / pk["bf16_sus"],
            "traffic": measured_traffic(dom),
            "traffic_note": "DRAM read+write bytes per launch (mean over the step's launches of this kind), "
                            "from profiles/roofline_traffic.json; null when the kernels changed since",
            "peak_note": f"bf16 dense burst ({pk['src']}); the sustained figure is {pk['bf16_sus']} TFLOP/s"
                         + ("; sw_power_cap was active during the timed region" if capped else ""),
            "flops_per_step": fl, "launches_per_step": kind_n[dom], "ms_per_step": ms_kind,
            "ms_per_step_eager": kind_ms[dom], "scale_to_graph_step": scale,
            "timing": "CUDA events around each launch on its stream during eager profiled steps, scaled so "
                      "that the kinds sum to the graph-timed ms_per_step"}


def pcie_rates(torch, dev, nbytes=512 << 20):
    """Pinned host <-> device copy rates of this machine (GB/s): each direction
    alone and both at once on two streams (best of three), the roofline of
    the end-to-end leg."""
    import time
    n = nbytes // 2
    h1 = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    h2 = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    d1 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    d2 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def h2d():
        with torch.cuda.stream(s1):
            d1.copy_(h1, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    def best(*fns):
        for f in fns:
            f()
        torch.cuda.synchronize()
        t = 1e9
        for _ in range(3):
            a = time.perf_counter()
            for f in fns:
                f()
            torch.cuda.synchronize()
            t = min(t, time.perf_counter() - a)
        return t
    th, td, tb = best(h2d), best(d2h), best(h2d, d2h)
    del h1, h2, d1, d2
    return {"h2d_gbs": nbytes / th / 1e9, "d2h_gbs": nbytes / td / 1e9, "both_gbs": 2 * nbytes / tb / 1e9}


def e2e_leg(qlora, torch, dev, P, G, M, r, world, steps, flops):
    """Same step through the C ABI with pinned host buffers: per step the H2D
    copy of every group's X and every projection's dY (in the order the step
    uses them), and the D2H copy of every Y, dA, dB and every group's dX, on
    two copy streams overlapping the compute stream."""
    hY = [torch.empty(d["Y"].shape, dtype=torch.bfloat16, pin_memory=True) for d in P]
    hdA = [torch.empty(d["dA"].shape, dtype=torch.float32, pin_memory=True) for d in P]
    hdB = [torch.empty(d["dB"].shape, dtype=torch.float32, pin_memory=True) for d in P]
    hdX = [torch.empty(g["dX"].shape, dtype=torch.bfloat16, pin_memory=True) for g in G]
    h2d = sum(P[g["idx"][0]]["hX"].numel() * 2 for g in G) + sum(d["hdY"].numel() * 2 for d in P)
    d2h = sum(d["Y"].numel() * 2 + d["dA"].numel() * 4 + d["dB"].numel() * 4 for d in P) + \
        sum(g["dX"].numel() * 2 for g in G)
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    comp = torch.cuda.current_stream()

    def after(stream_from, stream_to):
        ev = torch.cuda.Event()
        ev.record(stream_from)
        stream_to.wait_event(ev)

    def e2e_step():
        # inputs in the order the step consumes them: every X (forward, first
        # group first), then every dY in backward order (last group first),
        # so that each backward starts as soon as its own dY has arrived
        ev_x, ev_dy = [], [None] * len(G)
        for g in G:
            with torch.cuda.stream(s_h2d):
                g["X"].copy_(P[g["idx"][0]]["hX"], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_h2d)
                ev_x.append(e)
        for gi in reversed(range(len(G))):
            with torch.cuda.stream(s_h2d):
                for i in G[gi]["idx"]:
                    P[i]["dY"].copy_(P[i]["hdY"], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_h2d)
                ev_dy[gi] = e
        for gi, g in enumerate(G):
            comp.wait_event(ev_x[gi])
            qlora.qlora_group_fwd(g["X"], M, g["w"], g["A"], g["B"], r, g["s"], g["Y"], g["U"], g["ws"])
            after(comp, s_d2h)
            with torch.cuda.stream(s_d2h):
                for i in g["idx"]:
                    hY[i].copy_(P[i]["Y"], non_blocking=True)
        for gi in reversed(range(len(G))):
            g = G[gi]
            comp.wait_event(ev_dy[gi])
            qlora.qlora_group_bwd(g["X"], g["U"], M, g["w"], g["A"], g["B"], r, g["s"], g["dY"], g["dX"], g["dA"],
                                  g["dB"], g["ws"])
            if world > 1:
                dp.allreduce_adapter_grads(g["dA"] + g["dB"])
            after(comp, s_d2h)
            with torch.cuda.stream(s_d2h):
                hdX[gi].copy_(g["dX"], non_blocking=True)
                for i in g["idx"]:
                    hdA[i].copy_(P[i]["dA"], non_blocking=True)
                    hdB[i].copy_(P[i]["dB"], non_blocking=True)
        after(s_d2h, comp)

    e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for _ in range(steps):
        e2e_step()
    b.record(comp)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    pc = pcie_rates(torch, dev)
    copy_ms = max(h2d / pc["h2d_gbs"], d2h / pc["d2h_gbs"], (h2d + d2h) / pc["both_gbs"]) / 1e6
    return {"value": world * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pcie": {**pc, "copy_bound_ms_per_step": copy_ms, "frac": copy_ms / ms,
                     "note": "pinned copies of 512 MiB measured on this box; the step's host traffic at these "
                             "rates is its lower bound"},
            "note": "pinned host buffers; H2D of every group's X and every dY, D2H of every Y, dA, dB and every "
                    "group's dX, on two copy streams overlapping the compute stream; grouped calls"}


def bench_layer(qlora, torch, dev, pk, wl_id, steps):
    """A whole layer step (graph-timed) of another workload, grouped as the
    headline step, with its own per-kind times, and the same step as one
    call per projection."""
    wl, P, G = load_layer(qlora, torch, dev, wl_id)
    M, r = wl["M"], wl["r"]
    step = make_group_step(qlora, G, M, r, 1)
    ms = graph_time(torch, step, steps, 3)
    kms, kn = profile_kinds(qlora, torch, step, 3)
    ms_u = graph_time(torch, make_step(qlora, P, M, r, 1), steps, 3)
    _, kn_u = profile_kinds(qlora, torch, make_step(qlora, P, M, r, 1), 1)
    flops = step_flops(M, wl["projections"], r)
    v = flops / (ms * 1e-3) / 1e12
    out = {"workload": wl["name"], "M": M, "r": r, "alpha": wl["alpha"], "ms_per_step": ms, "value": v,
           "unit": "TFLOP/s", "pct_bf16_peak": v / pk["bf16"], "pct_bf16_peak_sustained": v / pk["bf16_sus"],
           "flops_per_step": flops, "groups": [g["name"] for g in G], "kernels_ms_per_step_eager": kms,
           "kernels_launches_per_step": kn,
           "roofline": roofline_of(kms, kn, ms, M, wl["projections"], r, pk, None),
           "ungrouped": {"ms_per_step": ms_u, "value": flops / (ms_u * 1e-3) / 1e12,
                         "launches_per_step": sum(kn_u.values())}}
    del P, G
    torch.cuda.empty_cache()
    return out


def bench_codec(qlora, torch, dev, pk):
    """14336 x 4096 quantize once + dequantize x100 (rotating over 6 copies of
    the packed weight, more than L2 holds, so reads come from HBM)."""
    _, cn, ck = synth.WORKLOADS[CODEC_WORKLOAD]["projections"][0]
    Wc = torch.from_numpy(synth.gaussian_bf16((cn, ck), 0.02, synth.seed_for(CODEC_WORKLOAD, "W")).view(np.int16))
    Wc = Wc.view(torch.bfloat16).to(dev)
    wc = qlora.alloc_nf4_weight(cn, ck, dev)
    wsc = qlora.workspace(qlora.qlora_nf4_quantize_workspace(cn, ck), dev)
    outc = torch.empty((cn, ck), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        qlora.qlora_nf4_quantize(Wc, wc, wsc)
        qlora.qlora_nf4_dequantize(wc, outc)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    qlora.qlora_nf4_quantize(Wc, wc, wsc)
    b.record()
    torch.cuda.synchronize()
    q_ms = a.elapsed_time(b)
    ncopy = 6
    wcs = [wc] + [qlora.alloc_nf4_weight(cn, ck, dev) for _ in range(ncopy - 1)]
    for x in wcs[1:]:
        x.codes.copy_(wc.codes); x.absmax_q.copy_(wc.absmax_q)
        x.absmax_scale.copy_(wc.absmax_scale); x.absmax_mean.copy_(wc.absmax_mean)
    outs = [outc, torch.empty_like(outc)]
    qlora.qlora_profile_start()
    torch.cuda.synchronize()
    a.record()
    for i in range(100):
        qlora.qlora_nf4_dequantize(wcs[i % ncopy], outs[i % 2])
    b.record()
    torch.cuda.synchronize()
    dq_prof_ms, dq_prof_n, _ = qlora.qlora_profile_stop()
    dq_ms = a.elapsed_time(b) / 100
    dq_kernel_ms = dq_prof_ms["dequant"] / max(1, dq_prof_n["dequant"])
    nel = cn * ck
    dq_bytes = nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4 + 2 * nel
    q_bytes = 2 * nel + nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4
    dq_gbs = dq_bytes / (dq_kernel_ms * 1e-3) / 1e9
    return {"workload": "nf4 codec 14336x4096 bf16 N(0,0.02)",
            "dequant": {"value": dq_gbs, "unit": "GB/s", "pct_hbm": dq_gbs / pk["hbm"],
                        "bytes_per_pass": dq_bytes, "ms_per_pass": dq_kernel_ms, "ms_per_call": dq_ms,
                        "l2": f"{ncopy} rotating copies of the packed weight (> L2)",
                        "roofline": {"bound": "hbm", "achieved": dq_gbs, "peak": pk["hbm"], "unit": "GB/s",
                                     "frac": dq_gbs / pk["hbm"], "traffic": measured_traffic("dequant"),
                                     "peak_note": f"HBM copy, {pk['src']}"}},
            "quantize": {"value": q_bytes / (q_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": q_ms, "bytes": q_bytes,
                         "pct_hbm": q_bytes / (q_ms * 1e-3) / 1e9 / pk["hbm"]}}


def bench_sweep(qlora, torch, dev, pk):
    """Token-count sweep on the gate projection 4096 -> 14336 (r = 16): the
    forward at every M, the backward for M >= 128. For M <= 16 the forward
    reads six rotating copies of the packed weight (more than L2 holds) and
    is reported as GB/s against the HBM roofline."""
    wl = synth.WORKLOADS[SWEEP]
    _, n, k = wl["projections"][0]
    r, scale = wl["r"], wl["scale"]
    dv = lambda h: torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    _, W, A, B, _, _ = synth.layer_inputs(SWEEP, 0, M=1)
    w0 = qlora.alloc_nf4_weight(n, k, dev)
    qlora.qlora_nf4_quantize(dv(W), w0, qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k), dev))
    Ad, Bd = dv(A), dv(B)
    del W
    rows = []
    for M in wl["M_sweep"]:
        # the same draws as synth.layer_inputs(SWEEP, 0, M) for X and dY
        X = synth.gaussian_bf16((M, k), 1.0, synth.seed_for(SWEEP, "X"))
        dY = synth.gaussian_bf16((M, n), 1.0, synth.seed_for(SWEEP, "dY")) if M >= 128 else None
        copies = 6 if M <= 16 else 1
        ws_ = [w0]
        for _ in range(copies - 1):
            x = qlora.alloc_nf4_weight(n, k, dev)
            x.codes.copy_(w0.codes); x.absmax_q.copy_(w0.absmax_q)
            x.absmax_scale.copy_(w0.absmax_scale); x.absmax_mean.copy_(w0.absmax_mean)
            ws_.append(x)
        Xd = dv(X)
        Y = torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        U = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
        wsb = qlora.workspace(max(qlora.qlora_linear_fwd_workspace(M, w0, r),
                                  qlora.qlora_linear_bwd_workspace(M, w0, r)), dev)
        it = [0]

        def fwd():
            w = ws_[it[0] % copies]
            it[0] += 1
            qlora.qlora_linear_fwd(Xd, M, w, Ad, Bd, r, scale, Y, U, wsb)

        reps = max(3, min(200, int(2e11 / max(1, M * n * k * 2))))
        if copies > 1:
            # one CUDA graph holding one call per weight copy, replayed: the
            # device time of the calls (eager launches from Python would be
            # bound by the host at these sizes); per-kernel times from eager
            # profiled calls
            def fwd_all():
                for _ in range(copies):
                    fwd()
            f_ms = graph_time(torch, fwd_all, max(3, reps // copies), 3) / copies
            torch.cuda.synchronize()
            qlora.qlora_profile_start()
            for _ in range(reps):
                fwd()
            torch.cuda.synchronize()
            pms, pn, _ = qlora.qlora_profile_stop()
        else:
            f_ms = graph_time(torch, fwd, reps, 3)
        f_fl = 2 * M * n * k + 2 * M * r * (n + k)
        row = {"M": M, "fwd_ms": f_ms, "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12}
        if M <= 16:
            wbytes = n * k // 2 + n * k // 64 + 4 * ((n * k // 64 + 255) // 256) + 4
            byts = wbytes + 2 * (M * k + M * n + r * k + n * r)
            gbs = byts / (f_ms * 1e-3) / 1e9
            row.update({"fwd_gbs": gbs, "fwd_pct_hbm": gbs / pk["hbm"], "fwd_bytes": byts,
                        "kernels_ms_per_call": {kk: v / reps for kk, v in pms.items() if pn[kk]},
                        "kernels_timing": "CUDA events around each launch during eager calls",
                        "l2": "6 rotating weight copies (> L2)"})
        if M >= 128:
            dYd = dv(dY)
            dX = torch.empty((M, k), dtype=torch.bfloat16, device=dev)
            dA = torch.empty((r, k), dtype=torch.float32, device=dev)
            dB = torch.empty((n, r), dtype=torch.float32, device=dev)

            def bwd():
                qlora.qlora_linear_bwd(dYd, Xd, U, M, w0, Ad, Bd, r, scale, dX, dA, dB, wsb)
            b_ms = graph_time(torch, bwd, reps, 3)
            b_fl = 2 * M * n * k + 4 * M * r * (n + k)
            row.update({"bwd_ms": b_ms, "bwd_tflops": b_fl / (b_ms * 1e-3) / 1e12,
                        "fwd_bwd_tflops": (4 * M * n * k + 6 * M * r * (n + k)) / ((f_ms + b_ms) * 1e-3) / 1e12})
            del dYd, dX
        rows.append(row)
        del Xd, ws_[1:], wsb
        torch.cuda.empty_cache()
    return {"workload": wl["name"] + ": gate 4096->14336 NF4+DQ, LoRA r=16 alpha=32", "rows": rows}


def bench_decode(qlora, torch, dev, pk, Ms=(1, 16)):
    """The 8B-shaped layer's forward at decode sizes (M = 1 and 16): the seven
    projections as grouped calls (q/k/v, o, gate/up, down) and as single
    calls, two copies of the layer's weights alternating (224 MB > L2),
    graph-replayed; GB/s counts the packed weights read (codes, absmax codes,
    scales) against the HBM roofline."""
    wl = synth.WORKLOADS[LAYER8B]
    r, scale = wl["r"], wl["scale"]
    projs = wl["projections"]
    groups = groups_of([{"name": nm} for nm, _, _ in projs])
    dv = lambda h: torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(dev)
    layers = []
    for copy in range(2):
        P = []
        for p, (nm, n, k) in enumerate(projs):
            _, W, A, B, _, _ = synth.layer_inputs(LAYER8B, p, M=1)
            w = qlora.alloc_nf4_weight(n, k, dev)
            qlora.qlora_nf4_quantize(dv(W), w, qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k), dev))
            P.append(dict(n=n, k=k, w=w, A=dv(A), B=dv(B)))
        layers.append(P)
    wbytes = sum(n * k // 2 + n * k // 64 + 4 * ((n * k // 64 + 255) // 256) + 4 for _, n, k in projs)
    rows = []
    for M in Ms:
        Xs = {k: torch.randn(M, k, device=dev).to(torch.bfloat16) for _, _, k in projs}
        for P in layers:
            for d in P:
                d["Y"] = torch.empty((M, d["n"]), dtype=torch.bfloat16, device=dev)
        U = torch.empty((M, 3 * r), dtype=torch.bfloat16, device=dev)
        U1 = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
        size = 0
        for P in layers:
            for d in P:
                size = max(size, qlora.qlora_linear_fwd_workspace(M, d["w"], r))
            for idx in groups:
                size = max(size, qlora.qlora_group_fwd_workspace(M, [P[i]["w"] for i in idx],
                                                                 [P[i]["A"] for i in idx], [P[i]["B"] for i in idx], r))
        ws = qlora.workspace(size, dev)

        def grouped():
            for P in layers:
                for idx in groups:
                    qlora.qlora_group_fwd(Xs[P[idx[0]]["k"]], M, [P[i]["w"] for i in idx], [P[i]["A"] for i in idx],
                                          [P[i]["B"] for i in idx], r, scale, [P[i]["Y"] for i in idx], U, ws)

        def single():
            for P in layers:
                for d in P:
                    qlora.qlora_linear_fwd(Xs[d["k"]], M, d["w"], d["A"], d["B"], r, scale, d["Y"], U1, ws)
        tg = graph_time(torch, grouped, 50, 3) / 2
        ts = graph_time(torch, single, 50, 3) / 2
        rows.append({"M": M, "layer_fwd_us_grouped": tg * 1e3, "layer_fwd_us_single": ts * 1e3,
                     "grouped_gbs": wbytes / (tg * 1e-3) / 1e9, "grouped_pct_hbm": wbytes / (tg * 1e-3) / 1e9 / pk["hbm"],
                     "single_gbs": wbytes / (ts * 1e-3) / 1e9})
        del ws, Xs
    del layers
    torch.cuda.empty_cache()
    return {"workload": wl["name"] + ": the seven projections' forward at decode sizes", "weight_bytes": wbytes,
            "rows": rows}


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def cpu_baseline():
    """The CPU oracle, as it stands, on bounded samples: the headline layer on
    CPU_SAMPLE_TOKENS tokens of every projection (all host cores, and one
    projection token on one thread), the codec, and the gate sweep at
    M <= 128. Rates need no extrapolation; the full-step time at M = 4096 is
    extrapolated linearly in the tokens and labelled so."""
    from oracle import oracle
    cores = host_cores()
    oracle.set_threads(cores)
    wl = synth.WORKLOADS[WORKLOAD]
    projs, r, M_full = wl["projections"], wl["r"], wl["M"]
    T = CPU_SAMPLE_TOKENS
    tot_t, tot_f = 0.0, 0
    one_thread = None
    for p, (name, n, k) in enumerate(projs):
        X, W, A, B, dY, s = synth.layer_inputs(WORKLOAD, p, M=T)
        Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
        del W
        t = time.perf_counter()
        oracle.linear_fwd(X, Wdq, A, B, s)
        oracle.linear_bwd(dY, X, Wdq, A, B, s)
        tot_t += time.perf_counter() - t
        tot_f += 4 * T * n * k + 6 * T * r * (n + k)
        if name == "gate":
            oracle.set_threads(1)
            t = time.perf_counter()
            oracle.linear_fwd(X[:1], Wdq, A, B, s)
            oracle.linear_bwd(dY[:1], X[:1], Wdq, A, B, s)
            t1 = time.perf_counter() - t
            oracle.set_threads(cores)
            one_thread = {"value": (4 * n * k + 6 * r * (n + k)) / t1 / 1e12, "unit": "TFLOP/s", "threads": 1,
                          "sample": "1 token of the 28672 x 8192 gate projection, forward + backward",
                          "seconds": t1}
    rate = tot_f / tot_t / 1e12
    full_flops = step_flops(M_full, projs, r)
    # codec: 14336 x 4096 quantize + dequantize
    _, cn, ck = synth.WORKLOADS[CODEC_WORKLOAD]["projections"][0]
    Wc = synth.gaussian_bf16((cn, ck), 0.02, synth.seed_for(CODEC_WORKLOAD, "W"))
    t = time.perf_counter()
    qw = oracle.nf4_quantize(Wc)
    tq = time.perf_counter() - t
    t = time.perf_counter()
    oracle.nf4_dequantize(qw)
    tdq = time.perf_counter() - t
    nel = cn * ck
    dq_bytes = nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4 + 2 * nel
    q_bytes = 2 * nel + nel // 2 + nel // 64 + 4 * ((nel // 64 + 255) // 256) + 4
    del Wc, qw
    # gate sweep at M <= 128 (the full problem at those token counts)
    sw = synth.WORKLOADS[SWEEP]
    _, n, k = sw["projections"][0]
    rs = sw["r"]
    X, W, A, B, dY, s = synth.layer_inputs(SWEEP, 0, M=128)
    Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
    sweep = []
    for M in (1, 16, 128):
        t = time.perf_counter()
        oracle.linear_fwd(X[:M], Wdq, A, B, s)
        tf = time.perf_counter() - t
        row = {"M": M, "fwd_tflops": (2 * M * n * k + 2 * M * rs * (n + k)) / tf / 1e12, "fwd_s": tf}
        if M == 128:
            t = time.perf_counter()
            oracle.linear_bwd(dY, X, Wdq, A, B, s)
            tb = time.perf_counter() - t
            row.update({"bwd_tflops": (2 * M * n * k + 4 * M * rs * (n + k)) / tb / 1e12, "bwd_s": tb})
        sweep.append(row)
    return {"value": rate, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{T} tokens of each of the 7 Llama-70B-shaped projections (r = 64), forward + backward "
                      f"(fp64 C loops, OpenMP on {cores} threads); {tot_t:.1f} s",
            "ms_per_step_extrapolated": 1e3 * full_flops / (rate * 1e12),
            "extrapolation": f"time of the full M = {M_full} step extrapolated linearly in the tokens "
                             f"from the {T}-token sample",
            "one_thread": one_thread,
            "codec": {"quantize_gbs": q_bytes / tq / 1e9, "dequant_gbs": dq_bytes / tdq / 1e9,
                      "quantize_s": tq, "dequant_s": tdq, "sample": "the full 14336 x 4096 codec workload"},
            "gate_sweep_M_le_128": sweep}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores on this arm's
    workload (the Llama-70B-shaped layer), each step a bounded sample: one
    token of one projection, forward + backward, round robin over the seven."""
    if rank != 0:
        return
    from oracle import oracle
    cores = host_cores()
    oracle.set_threads(cores)
    w = synth.WORKLOADS[WORKLOAD]
    projs, r = w["projections"], w["r"]
    prep = []
    for p in range(len(projs)):
        X, W, A, B, dY, s = synth.layer_inputs(WORKLOAD, p, M=1)
        prep.append((X, oracle.nf4_dequantize(oracle.nf4_quantize(W)), A, B, dY, s, projs[p]))
        del W

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
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(w), "M": w["M"], "r": r,
                   "sample": "1 token of one projection per step (round robin over q,k,v,o,gate,up,down)"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "1 token of one projection (round robin over q,k,v,o,gate,up,down) per step"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--prof-steps", type=int, default=3)
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other layers, the codec and the M sweep")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
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
    props = torch.cuda.get_device_properties(dev)

    wl, P, G = load_layer(qlora, torch, dev, WORKLOAD, pinned=True)
    projs, M, r = wl["projections"], wl["M"], wl["r"]
    stream = torch.cuda.current_stream()
    step = make_group_step(qlora, G, M, r, world)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    qlora.qlora_check_device_status(stream)
    barrier()

    # The timed region replays one CUDA graph of the step (the library's calls
    # allocate and synchronize nothing, so they capture as they are), or
    # launches the step eagerly with --no-graph.
    graph = capture(torch, step) if not args.no_graph and world == 1 else None
    if graph is not None:
        qlora.qlora_check_device_status(stream)
    run_step = graph.replay if graph is not None else step

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        barrier()
        clk.mark_start()
        ev0.record()
        for _ in range(args.steps):
            run_step()
        ev1.record()
        barrier()
        clk.mark_end()
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

    kind_ms, kind_n = profile_kinds(qlora, torch, step, max(1, args.prof_steps))
    launches = sum(kind_n.values()) * args.steps
    roof = roofline_of(kind_ms, kind_n, ms_step, M, projs, r, pk, clocks)
    e2e = e2e_leg(qlora, torch, dev, P, G, M, r, world, args.e2e_steps, flops)
    timed_region = "CUDA graph of one step replayed" if graph is not None else "eager launches"
    ungrouped = None
    if world == 1 and not args.no_extra:
        ustep = make_step(qlora, P, M, r, 1)
        # same number of graph-replayed steps as the headline, then the grouped
        # step once more right after, so the two see the same clock conditions
        ms_u = graph_time(torch, ustep, args.steps, 3)
        ms_g = graph_time(torch, step, args.steps, 3)
        _, kn_u = profile_kinds(qlora, torch, ustep, 1)
        ungrouped = {"ms_per_step": ms_u, "value": flops / (ms_u * 1e-3) / 1e12,
                     "launches_per_step": sum(kn_u.values()),
                     "grouped_ms_per_step_after": ms_g,
                     "note": "the same step as seven single-layer calls (each projection reads X itself and "
                             "returns its own dX), timed like the headline; grouped_ms_per_step_after times the "
                             "grouped step again right after it"}
    del P, G, graph
    torch.cuda.empty_cache()

    extra = {}
    if rank == 0 and world == 1 and not args.no_extra:
        extra["llama8b_layer"] = bench_layer(qlora, torch, dev, pk, LAYER8B, 100)
        extra["single_layer"] = bench_layer(qlora, torch, dev, pk, SINGLE, 200)
        extra["codec"] = bench_codec(qlora, torch, dev, pk)
        extra["gate_sweep"] = bench_sweep(qlora, torch, dev, pk)
        extra["decode_layer"] = bench_decode(qlora, torch, dev, pk)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "pct_bf16_peak": value / world / pk["bf16"], "pct_bf16_peak_sustained": value / world / pk["bf16_sus"],
            "config": {"workload": workload_name(wl),
                       "M": M, "r": r, "alpha": wl["alpha"], "projections": [[n_, k_] for _, n_, k_ in projs],
                       "flops_per_step": flops, "parallelism": f"dp{world}",
                       "l2": "inputs larger than L2 (several GB touched per step)",
                       "l2_cache_bytes": int(props.L2_cache_size), "sm_count": props.multi_processor_count},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "kernels_ms_per_step_eager": kind_ms,
            "kernels_launches_per_step": kind_n,
            "ungrouped": ungrouped,
            "timed_region": timed_region,
            "clocks": clocks,
            **extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
