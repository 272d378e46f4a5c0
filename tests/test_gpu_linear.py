"""GPU parity of the LoRA linear layer, forward and backward, against the CPU
oracle on the identically dequantized weights.

Bar: relative Frobenius error <= 5e-3 per output tensor (Y, U, dX, dA, dB).
The GPU accumulates in fp32 over bf16 operands and rounds Y and dX to bf16
(relative rounding error up to 2^-9 per element, about 1.1e-3 in Frobenius
norm); the LoRA side path runs through s*U or s*V rounded to bf16. The oracle
accumulates in fp64.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


def make(M, N, K, r, seed, a_std=None, w_zero=False):
    X = synth.gaussian_bf16((M, K), 1.0, seed)
    W = np.zeros((N, K), np.uint16) if w_zero else synth.gaussian_bf16((N, K), 0.02, seed + 1)
    A = synth.gaussian_bf16((r, K), a_std if a_std else 1.0 / K, seed + 2)
    B = synth.gaussian_bf16((N, r), 0.01, seed + 3)
    dY = synth.gaussian_bf16((M, N), 1.0, seed + 4)
    return X, W, A, B, dY


def run_and_check(g, oracle, M, N, K, r, scale, seed, **kw):
    X, W, A, B, dY = make(M, N, K, r, seed, **kw)
    qw = oracle.nf4_quantize(W)
    Wdq = oracle.nf4_dequantize(qw)
    w = g.weight_from_oracle(qw)
    Y, U = g.fwd(X, w, A, B, r, scale)
    Yref, Uref = oracle.linear_fwd(X, Wdq, A, B, scale)
    errs = {"Y": g.rel_fro(g.host_f64_bf16(Y), Yref), "U": g.rel_fro(g.host_f64_bf16(U), Uref)}
    dX, dA, dB = g.bwd(dY, X, U, w, A, B, r, scale)
    dXr, dAr, dBr = oracle.linear_bwd(dY, X, Wdq, A, B, scale)
    errs["dX"] = g.rel_fro(g.host_f64_bf16(dX), dXr)
    errs["dA"] = g.rel_fro(dA.cpu().numpy(), dAr)
    errs["dB"] = g.rel_fro(dB.cpu().numpy(), dBr)
    # recomputing U inside the backward gives the same gradients
    dX2, dA2, dB2 = g.bwd(dY, X, None, w, A, B, r, scale)
    errs["dB(recompute U)"] = g.rel_fro(dB2.cpu().numpy(), dBr)
    errs["dX(recompute U)"] = g.rel_fro(g.host_f64_bf16(dX2), dXr)
    for k, v in errs.items():
        assert v <= TOL, (k, v, errs)
    return errs


@pytest.mark.parametrize("M,N,K,r,scale", [
    (256, 1024, 1024, 8, 2.0),     # the single-layer workload
    (77, 192, 320, 5, 2.0),        # ragged M, N; r not a multiple of 8
    (1, 320, 256, 16, 2.0),        # one token
    (16, 1000, 512, 16, 2.0),
    (130, 256, 640, 64, 0.25),
    (64, 128, 128, 128, 0.5),      # largest rank
    (300, 448, 384, 1, 4.0),       # smallest rank
    (512, 1024, 2048, 16, 2.0),    # tensor-core path, full tiles
    (200, 520, 1088, 64, 0.25),    # tensor-core path: ragged M, N and K tiles
    (128, 256, 4096, 72, 0.5),     # two LoRA k-steps
    (20, 100, 192, 8, 2.0),        # few tokens, N not a multiple of 8
    (70, 100, 192, 8, 2.0),        # tensor-core forward, CUDA-core backward (N % 8 != 0)
    (32, 2048, 1024, 16, 2.0),     # largest few-token forward (four 8-token tiles)
    (24, 512, 14336, 16, 2.0),     # few tokens, longest K of the table
    # fused-GEMM schedules on 74 CTA pairs (tiles of 512 x 256):
    (2048, 9728, 128, 16, 2.0),    # forward: 152 tiles, one data-parallel round + stream-K over 78
    (2048, 128, 9728, 16, 2.0),    # dX: the same split on the backward
    (2148, 4000, 192, 8, 1.0),     # stream-K over 80 tiles, 100-row last row tile, ragged N
    (4708, 2048, 128, 8, 1.0),     # ten row tiles: two bands of the tile order, the second partial
    # few-token forward (M <= 16, K a multiple of 256; tasks of 32 rows x 256 k,
    # one pipeline per warp, row tiles shared between warps finished by the last):
    (1, 4096, 1024, 16, 2.0),      # one token, 512 tasks on 512 warps: four warps per row tile
    (16, 14336, 4096, 16, 2.0),    # the gate projection at 16 tokens
    (5, 1000, 2048, 8, 2.0),       # ragged N (last row tile of 8 rows), r % 8 == 0
    (9, 96, 4096, 5, 2.0),         # 48 tasks on 48 warps: every row tile shared by 16 warps, odd r
    (2, 33, 1024, 16, 2.0),        # a row tile with one valid row
    (1, 1, 1024, 3, 2.0),          # a single weight row
    (12, 520, 3072, 64, 0.25),     # rank 64: four LoRA steps in the finishing
    (3, 700, 256, 16, 2.0),        # K = 256: one task per row tile, every tile finished by its own warp
    (4, 256, 1024, 128, 0.5),      # largest rank: eight LoRA steps in the finishing, 128 sU CTAs a token
    (16, 64, 512, 128, 0.5),       # sixteen tokens at the largest rank
    (16, 4096, 14336, 16, 1.0),    # 8B down projection: ~20 warps per row tile (several slot chunks)
])
def test_fwd_bwd_parity(g, oracle, M, N, K, r, scale):
    run_and_check(g, oracle, M, N, K, r, scale, seed=3000 + M + N + r)


@pytest.mark.parametrize("M,N,K,r", [(256, 1024, 1024, 8), (33, 200, 192, 16), (8, 512, 2048, 16)])
def test_lora_only(g, oracle, M, N, K, r):
    # W == 0 quantizes to code 7 everywhere and dequantizes to exact zeros, so
    # Y is the LoRA term alone and dX is its gradient alone.
    run_and_check(g, oracle, M, N, K, r, 2.0, seed=4000 + M, w_zero=True)


def test_strong_adapter(g, oracle):
    # the single-layer workload with A ~ N(0, 1/32): the LoRA term is a visible
    # share of Y
    run_and_check(g, oracle, 256, 1024, 1024, 8, 2.0, seed=5000, a_std=1.0 / 32)


def test_empty_batch(g, oracle):
    import torch
    from bit_quantized_lora_double_b300 import qlora
    X, W, A, B, dY = make(4, 128, 128, 8, 6000)
    w = g.quantize(W)
    Y = torch.full((1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    qlora.qlora_linear_fwd(g.dev_bf16(X), 0, w, g.dev_bf16(A), g.dev_bf16(B), 8, 2.0, Y, None, None)
    assert torch.all(Y == 7.0)
    dA = torch.full((8, 128), 3.0, device="cuda")
    dB = torch.full((128, 8), 3.0, device="cuda")
    dX = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    qlora.qlora_linear_bwd(g.dev_bf16(dY), g.dev_bf16(X), None, 0, w, g.dev_bf16(A), g.dev_bf16(B), 8, 2.0, dX, dA,
                           dB, None)
    torch.cuda.synchronize()
    assert torch.all(dA == 0) and torch.all(dB == 0)
