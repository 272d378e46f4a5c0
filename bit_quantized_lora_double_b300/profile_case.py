"""Runs one NF4-LoRA projection (quantize, then forward + backward) a few
times through the C ABI and prints per-kernel-kind device times. Meant as a
small, self-contained case to put under a profiler:

  python -m bit_quantized_lora_double_b300.profile_case --projection gate --M 2048 --reps 3
  python -m bit_quantized_lora_double_b300.profile_case --projection gate --M 1 --fwd-only
  python -m bit_quantized_lora_double_b300.profile_case --codec --reps 3   # 14336 x 4096 quantize + dequantize
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
    args = ap.parse_args()

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
    print(json.dumps({"projection": args.projection, "M": M, "N": n, "K": k, "r": r, "reps": args.reps,
                      "ms_per_rep": {kk: v / args.reps for kk, v in ms.items() if cnt[kk]},
                      "launches_per_rep": {kk: v // args.reps for kk, v in cnt.items() if v}}))


if __name__ == "__main__":
    main()
