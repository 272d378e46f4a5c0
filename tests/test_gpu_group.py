"""GPU parity of projection groups (several LoRA linears sharing X, one call).

The grouped forward and backward are checked against the oracle's group
functions (each projection's Y_g, U_g, dA_g, dB_g, and dX summed over the
projections) with the linear layer's bar: relative Frobenius error <= 5e-3
per output tensor. Shapes cover the tensor-core paths (one fused GEMM over all
projections' columns, or rows for dX), ragged N and M, groups of one to four,
the few-token paths (the forward as one launch over the group's row tiles, the
backward projection by projection), U recomputed in the backward,
adapters given back to back or apart, and the batched side-path launches (all
V passes of a group in one launch; dA with every dB in one launch when their
ranks take the same number of 64-wide tiles, up to five problems).
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import qlora, synth

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


def run_group(g, oracle, M, Ns, K, r, scale, seed, save_u=True, packed=False, rows=None):
    import torch
    n = len(Ns)
    X = synth.gaussian_bf16((M, K), 1.0, seed)
    Ws = [synth.gaussian_bf16((N, K), 0.02, seed + 10 * i + 1) for i, N in enumerate(Ns)]
    As = [synth.gaussian_bf16((r, K), 1.0 / K, seed + 10 * i + 2) for i in range(n)]
    Bs = [synth.gaussian_bf16((N, r), 0.01, seed + 10 * i + 3) for i, N in enumerate(Ns)]
    dYs = [synth.gaussian_bf16((M, N), 1.0, seed + 10 * i + 4) for i, N in enumerate(Ns)]
    qws = [oracle.nf4_quantize(W) for W in Ws]
    Wdqs = [oracle.nf4_dequantize(q) for q in qws]
    wts = [g.weight_from_oracle(q) for q in qws]
    Xd = g.dev_bf16(X)
    if packed:
        # adapters and dA back to back: the library uses them in place
        Acat = g.dev_bf16(np.vstack(As))
        Ad = [Acat[i * r:(i + 1) * r] for i in range(n)]
        dAcat = torch.empty((n * r, K), dtype=torch.float32, device="cuda")
        dAs = [dAcat[i * r:(i + 1) * r] for i in range(n)]
    else:
        Ad = [g.dev_bf16(A) for A in As]
        dAs = [torch.empty((r, K), dtype=torch.float32, device="cuda") for _ in range(n)]
    Bd = [g.dev_bf16(B) for B in Bs]
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for N in Ns]
    U = torch.empty((M, n * r), dtype=torch.bfloat16, device="cuda") if save_u else None
    wsf = qlora.workspace(qlora.qlora_group_fwd_workspace(M, wts, Ad, Bd, r))
    qlora.qlora_group_fwd(Xd, M, wts, Ad, Bd, r, scale, Ys, U, wsf)
    dYd = [g.dev_bf16(d) for d in dYs]
    dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dBs = [torch.empty((N, r), dtype=torch.float32, device="cuda") for N in Ns]
    wsb = qlora.workspace(qlora.qlora_group_bwd_workspace(M, wts, Ad, Bd, r))
    qlora.qlora_group_bwd(Xd, U, M, wts, Ad, Bd, r, scale, dYd, dX, dAs, dBs, wsb)
    torch.cuda.synchronize()
    qlora.qlora_check_device_status()

    ri = None if rows is None else torch.from_numpy(rows).cuda()
    sel = (lambda t: t) if rows is None else (lambda t: t.index_select(0, ri))
    outs = oracle.group_fwd(X, Wdqs, As, Bs, scale, rows=rows)
    dXr, grads = oracle.group_bwd(dYs, X, Wdqs, As, Bs, scale, rows=rows)
    errs = {}
    for i in range(n):
        Yr, Ur = outs[i]
        errs[f"Y{i}"] = g.rel_fro(g.host_f64_bf16(sel(Ys[i])), Yr)
        if save_u:
            errs[f"U{i}"] = g.rel_fro(g.host_f64_bf16(U[:, i * r:(i + 1) * r]), Ur)
        errs[f"dA{i}"] = g.rel_fro(dAs[i].cpu().numpy(), grads[i][0])
        errs[f"dB{i}"] = g.rel_fro(dBs[i].cpu().numpy(), grads[i][1])
    errs["dX"] = g.rel_fro(g.host_f64_bf16(sel(dX)), dXr)
    for k, v in errs.items():
        assert v <= TOL, (k, v, errs)
    return errs


@pytest.mark.parametrize("M,Ns,K,r,scale,save_u,packed", [
    (384, [1024, 256, 256], 1024, 16, 2.0, True, False),    # q/k/v-shaped, tensor cores
    (384, [1024, 256, 256], 1024, 16, 2.0, True, True),     # adapters back to back
    (200, [2048, 2048], 512, 8, 1.0, False, False),         # gate/up-shaped, ragged M, U recomputed
    (130, [296, 136], 256, 16, 0.5, True, False),           # N not multiples of 64 or 256
    (256, [512, 384, 256, 128], 512, 64, 0.25, True, True), # four projections, r = 64
    (200, [256, 128, 384, 128], 512, 16, 1.0, False, False),  # four, r = 16: dA and the four dB in one launch
    (96, [640], 768, 24, 2.0, True, False),                 # a group of one, r = 24
])
def test_group_parity(g, oracle, M, Ns, K, r, scale, save_u, packed):
    run_group(g, oracle, M, Ns, K, r, scale, seed=M + len(Ns), save_u=save_u, packed=packed)


@pytest.mark.parametrize("M,Ns,K,r,save_u", [
    (5, [1024, 256, 256], 1024, 16, True),    # few-token forward (one launch over the group), CUDA-core backward
    (16, [512, 512], 2048, 8, False),         # two 8-token tiles, U recomputed
    (3, [100, 36, 520, 64], 512, 16, True),   # four projections, row tiles ragged at every projection's end
    (1, [4096, 1024, 1024], 4096, 16, True),  # the 8B layer's q/k/v at one token
    (24, [300, 100], 320, 8, True),           # small-M forward; N % 8 != 0
    (70, [300, 96], 256, 16, True),           # tensor-core forward, CUDA-core backward (N % 8)
])
def test_group_few_tokens(g, oracle, M, Ns, K, r, save_u):
    run_group(g, oracle, M, Ns, K, r, 2.0, seed=7 * M, save_u=save_u)


@pytest.mark.slow
def test_group_llama8b_qkv(g, oracle):
    # the 8B layer's q/k/v (4096, 1024, 1024 x 4096) at M = 2048, r = 16,
    # on 128 sampled token rows
    rows = np.sort(np.random.default_rng(5).choice(2048, 128, replace=False))
    run_group(g, oracle, 2048, [4096, 1024, 1024], 4096, 16, 2.0, seed=2048, rows=rows)


def test_group_matches_single_calls(g, oracle):
    """The group's outputs against the single-layer calls on the same inputs:
    the same arithmetic per projection up to fp32 summation order."""
    import torch
    M, Ns, K, r, s = 256, [768, 256], 512, 16, 2.0
    X = synth.gaussian_bf16((M, K), 1.0, 1)
    Ws = [synth.gaussian_bf16((N, K), 0.02, 2 + i) for i, N in enumerate(Ns)]
    As = [synth.gaussian_bf16((r, K), 1.0 / K, 5 + i) for i in range(2)]
    Bs = [synth.gaussian_bf16((N, r), 0.01, 8 + i) for i, N in enumerate(Ns)]
    wts = [g.quantize(W) for W in Ws]
    Ad, Bd = [g.dev_bf16(A) for A in As], [g.dev_bf16(B) for B in Bs]
    Ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for N in Ns]
    ws = qlora.workspace(qlora.qlora_group_fwd_workspace(M, wts, Ad, Bd, r))
    qlora.qlora_group_fwd(g.dev_bf16(X), M, wts, Ad, Bd, r, s, Ys, None, ws)
    torch.cuda.synchronize()
    for i in range(2):
        Y1, _ = g.fwd(X, wts[i], As[i], Bs[i], r, s)
        assert g.rel_fro(g.host_f64_bf16(Ys[i]), g.host_f64_bf16(Y1)) <= 2e-3
