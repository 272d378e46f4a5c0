"""Runs one NF4-LoRA projection (quantize, then forward + backward) a few
times through the C ABI and prints per-kernel-kind device times. Meant as a
small, self-contained case to put under a profiler:

  python -m bit_quantized_lora_double_b300.profile_case --projection gate --M 2048 --reps 3
  python -m bit_quantized_lora_double_b300.profile_case --projection gate --M 1 --fwd-only
  python -m bit_quantized_lora_double_b300.profile_case --codec --reps 3   # 14336 x 4096 quantize + dequantize
  python -m bit_quantized_lora_double_b300.profile_case --workload 3 --projection q --M 4096 --stamps fwd

--stamps fwd|dx builds the diagnostic library (the fused GEMM records
globaltimer stamps of its first CTA pair; no work is skipped), runs the
projection and prints the timeline of the last forward (or dX) GEMM launch:
k-step period, TMA latency as the decoders see it, decode time, how early the
decoded tiles are ready, the MMA issue time, and the drain at tile ends.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from bit_quantized_lora_double_b300 import qlora, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--projection", default="gate")
    ap.add_argument("--M", type=int, default=2048)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--codec", action="store_true")
    ap.add_argument("--stamps", choices=["fwd", "dx", "few"], default=None)
    args = ap.parse_args()
    if args.stamps:
        from bit_quantized_lora_double_b300 import _build
        qlora._LIB_PATH = _build.build(stamps=True)

    def dev(h):
        return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).view(torch.bfloat16).cuda()

    if args.codec:
        _, n, k = synth.WORKLOADS[2]["projections"][0]
        W = dev(synth.gaussian_bf16((n, k), 0.02, synth.seed_for(2, "W")))
        w = qlora.alloc_nf4_weight(n, k)
        ws = qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k))
        out = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        qlora.qlora_profile_start()
        for _ in range(args.reps):
            qlora.qlora_nf4_quantize(W, w, ws)
            qlora.qlora_nf4_dequantize(w, out)
        torch.cuda.synchronize()
        ms, cnt, total = qlora.qlora_profile_stop()
        print(json.dumps({"codec": [n, k], "reps": args.reps,
                          "ms_per_rep": {kk: v / args.reps for kk, v in ms.items() if cnt[kk]}}))
        return

    wl = synth.WORKLOADS[args.workload]
    names = [p[0] for p in wl["projections"]]
    p = names.index(args.projection)
    _, n, k = wl["projections"][p]
    r, M = wl["r"], args.M
    X, W, A, B, dY, s = synth.layer_inputs(args.workload, p, M=M)
    w = qlora.alloc_nf4_weight(n, k)
    qlora.qlora_nf4_quantize(dev(W), w, qlora.workspace(qlora.qlora_nf4_quantize_workspace(n, k)))
    Xd, Ad, Bd, dYd = dev(X), dev(A), dev(B), dev(dY)
    Y = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    U = torch.empty((M, r), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((M, k), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((r, k), dtype=torch.float32, device="cuda")
    dB = torch.empty((n, r), dtype=torch.float32, device="cuda")
    ws = qlora.workspace(max(qlora.qlora_linear_fwd_workspace(M, w, r), qlora.qlora_linear_bwd_workspace(M, w, r)))
    torch.cuda.synchronize()
    qlora.qlora_profile_start()
    for _ in range(args.reps):
        qlora.qlora_linear_fwd(Xd, M, w, Ad, Bd, r, s, Y, U, ws)
        if not args.fwd_only:
            qlora.qlora_linear_bwd(dYd, Xd, U, M, w, Ad, Bd, r, s, dX, dA, dB, ws)
    torch.cuda.synchronize()
    ms, cnt, total = qlora.qlora_profile_stop()
    qlora.qlora_check_device_status()
    if args.stamps == "few":
        qlora.qlora_linear_fwd(Xd, M, w, Ad, Bd, r, s, Y, U, ws)
        torch.cuda.synchronize()
        print_few_timeline()
    elif args.stamps:
        if args.stamps == "fwd":
            qlora.qlora_linear_fwd(Xd, M, w, Ad, Bd, r, s, Y, U, ws)
            seg = qlora.qlora_debug_gemm_segments(M, n, k // 64, (r + 63) // 64, 74)
        else:
            qlora.qlora_linear_bwd(dYd, Xd, U, M, w, Ad, Bd, r, s, dX, dA, dB, ws)
            seg = qlora.qlora_debug_gemm_segments(M, k, (n + 63) // 64, (r + 63) // 64, 74)
        torch.cuda.synchronize()
        print_timeline(seg)
    print(json.dumps({"projection": args.projection, "M": M, "N": n, "K": k, "r": r, "reps": args.reps,
                      "ms_per_rep": {kk: v / args.reps for kk, v in ms.items() if cnt[kk]},
                      "launches_per_rep": {kk: v // args.reps for kk, v in cnt.items() if v}}))


def print_timeline(seg):
    """Summary of the diagnostic GEMM timeline of the first CTA pair."""
    import ctypes
    L = qlora.lib()
    L.qlora_debug_gemm_stamps.argtypes = [ctypes.c_void_p]
    L.qlora_debug_gemm_stamps.restype = ctypes.c_int
    h = np.zeros(8 * 4096, np.uint64)
    assert L.qlora_debug_gemm_stamps(h.ctypes.data) == 0
    h = h.reshape(8, 4096).astype(np.int64)
    rec = seg[4]
    mine = rec[rec[:, 0] == 0]  # pair 0's segments
    steps, tiles = int(mine[:, 5].sum()), len(mine)
    iss, fl, dec, rdy, cm, pdec = (h[i, :steps] for i in (0, 1, 2, 3, 4, 7))
    q = lambda a, p: float(np.percentile(a, p))
    per = np.diff(cm) / 1e3
    late = np.maximum(dec, pdec)[1:] > cm[:-1]
    out = {
        "pair0_steps": steps, "pair0_segments": tiles,
        "span_us": (cm[-1] - iss[0]) / 1e3,
        "step_us": {"median": q(per, 50), "mean": float(per.mean()), "p90": q(per, 90)},
        "tma_landed_after_issue_us": {"median": q((fl - iss) / 1e3, 50), "p90": q((fl - iss) / 1e3, 90)},
        "decode_us": {"median": q((dec - fl) / 1e3, 50), "p90": q((dec - fl) / 1e3, 90)},
        "decoded_ahead_of_issuer_us_median": q((rdy - dec) / 1e3, 50),
        "steps_decoded_late_pct": 100.0 * float(late.mean()),
        "mma_issue_us_median": q((cm - rdy) / 1e3, 50),
        "issuer_wait_between_steps_us_median": q((rdy[1:] - cm[:-1]) / 1e3, 50),
        "tile_drain_us": [float((h[6, t] - h[5, t]) / 1e3) for t in range(tiles) if h[6, t] > h[5, t]],
    }
    print(json.dumps({"gemm_timeline": out}))


def print_few_timeline():
    """Summary of the few-token forward's per-warp timeline (us from the
    earliest warp's entry): percentiles over warps of each event."""
    import ctypes
    L = qlora.lib()
    L.qlora_debug_few_stamps.argtypes = [ctypes.c_void_p]
    L.qlora_debug_few_stamps.restype = ctypes.c_int
    h = np.zeros(148 * 16 * 16, np.uint64)  # at least the device array
    assert L.qlora_debug_few_stamps(h.ctypes.data) == 0
    h = h.reshape(-1, 16).astype(np.int64)
    last = h[:, 0].max()
    h = h[(h[:, 0] > 0) & (h[:, 0] > last - 10**6) & (h[:, 14] >= h[:, 0])]
    t0 = h[:, 0].min()
    rel = lambda c: (h[:, c] - t0) / 1e3
    pct = lambda a: {p: round(float(np.percentile(a, p)), 2) for p in (0, 10, 50, 90, 100)}
    out = {"warps": int(len(h)), "entry": pct(rel(0)), "after_start_barrier": pct(rel(1))}
    for i in range(4):
        ok = h[:, 2 + 2 * i] >= h[:, 0]
        if ok.sum() == 0:
            break
        out[f"task{i}_landed"] = pct(rel(2 + 2 * i)[ok])
        out[f"task{i}_decode_us"] = pct(((h[:, 3 + 2 * i] - h[:, 2 + 2 * i]) / 1e3)[ok])
    for e in range(2):
        ok = h[:, 11 + 2 * e] >= h[:, 10 + 2 * e]
        ok &= h[:, 10 + 2 * e] >= h[:, 0]
        if ok.sum():
            out[f"tile_end{e}_us"] = pct(((h[:, 11 + 2 * e] - h[:, 10 + 2 * e]) / 1e3)[ok])
    out["stream_done"] = pct(rel(14))
    out["warps_finishing_tiles"] = int((h[:, 15] > 0).sum())
    print(json.dumps({"few_timeline": out}))


if __name__ == "__main__":
    main()
