"""Data-parallel decomposition on CPU with two gloo ranks: every rank takes
its token shard, computes the backward with the oracle, and the all-reduced
adapter gradients equal the full-batch ones; the per-token outputs are the
matching rows of the full-batch outputs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from bit_quantized_lora_double_b300 import dp, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, M, N, K, r, scale, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import oracle
        X = synth.gaussian_bf16((M, K), 1.0, 71)
        W = synth.gaussian_bf16((N, K), 0.02, 72)
        A = synth.gaussian_bf16((r, K), 1.0 / 16, 73)
        B = synth.gaussian_bf16((N, r), 0.05, 74)
        dY = synth.gaussian_bf16((M, N), 1.0, 75)
        Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
        a, b = dp.token_shard(M, rank, world)
        Y, _ = oracle.linear_fwd(X[a:b], Wdq, A, B, scale)
        dX, dA, dB = oracle.linear_bwd(dY[a:b], X[a:b], Wdq, A, B, scale)
        g = [torch.from_numpy(np.ascontiguousarray(dA)), torch.from_numpy(np.ascontiguousarray(dB))]
        dp.allreduce_adapter_grads(g)
        out[rank] = (a, b, Y, dX, g[0].numpy(), g[1].numpy())
    finally:
        dist.destroy_process_group()


def test_token_shards_cover_exactly():
    for M in (0, 1, 7, 64, 1000):
        for world in (1, 2, 3, 8):
            spans = [dp.token_shard(M, rk, world) for rk in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == M
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1


def test_two_gloo_ranks_match_full_batch(oracle):
    M, N, K, r, scale = 37, 48, 128, 4, 2.0
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), M, N, K, r, scale, out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    X = synth.gaussian_bf16((M, K), 1.0, 71)
    W = synth.gaussian_bf16((N, K), 0.02, 72)
    A = synth.gaussian_bf16((r, K), 1.0 / 16, 73)
    B = synth.gaussian_bf16((N, r), 0.05, 74)
    dY = synth.gaussian_bf16((M, N), 1.0, 75)
    Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
    Y, _ = oracle.linear_fwd(X, Wdq, A, B, scale)
    dX, dA, dB = oracle.linear_bwd(dY, X, Wdq, A, B, scale)
    for rank in (0, 1):
        a, b, Yr, dXr, dAr, dBr = res[rank]
        np.testing.assert_allclose(Yr, Y[a:b], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dXr, dX[a:b], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dAr, dA, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dBr, dB, rtol=1e-10, atol=1e-12)
