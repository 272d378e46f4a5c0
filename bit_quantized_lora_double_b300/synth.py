"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no arithmetic of the method: it only draws Gaussian numbers
and rounds them to bf16 bit patterns, so the GPU path and the CPU oracle can be
fed the same bytes.

Recipe: numpy ``Generator(PCG64(seed))`` draws float32 standard normals
(``standard_normal(dtype=float32)``), multiplies them by the float32 std
(round to nearest) and rounds the products to bf16 with round-to-nearest-even
on the bit pattern. Seeds are
``20261202 + 100 * workload + tensor`` with tensor X=0, W=1, A=2, B=3, dY=4;
projection p of a multi-projection workload adds ``10 * p``.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
TENSOR = {"X": 0, "W": 1, "A": 2, "B": 3, "dY": 4}


def seed_for(workload: int, tensor: str, projection: int = 0) -> int:
    return SEED_BASE + 100 * workload + 10 * projection + TENSOR[tensor]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    # finite inputs stay below 0xFF800000 + 0x8000, so uint32 does not wrap
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def gaussian_bf16(shape, std: float, seed: int, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std^2) draws as bf16 bit patterns, generated in chunks to bound host memory."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = f32_to_bf16_bits(rng.standard_normal(m, dtype=np.float32) * np.float32(std))
    return out.reshape(shape)


def zeros_bf16(shape) -> np.ndarray:
    return np.zeros(shape, np.uint16)


# Workload shapes (projections are (name, N out, K in)).
LLAMA8B_LAYER = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
                 ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]
LLAMA70B_LAYER = [("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
                  ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)]

WORKLOADS = {
    # id: dict(projections, M, r, LoRA alpha and scale = alpha / r, A std, B std, W std)
    0: dict(name="single-1024x1024-M256-r8", projections=[("single", 1024, 1024)], M=256, r=8,
            alpha=16.0, scale=2.0, a_std="1/K", b_std=0.01, w_std=0.02),
    1: dict(name="llama3.1-8b-layer-M2048-r16", projections=LLAMA8B_LAYER, M=2048, r=16,
            alpha=32.0, scale=2.0, a_std="1/K", b_std=0.01, w_std=0.02),
    2: dict(name="nf4-codec-14336x4096", projections=[("gate", 14336, 4096)], M=0, r=0,
            alpha=0.0, scale=0.0, a_std="1/K", b_std=0.0, w_std=0.02),
    3: dict(name="llama-70b-layer-M4096-r64", projections=LLAMA70B_LAYER, M=4096, r=64,
            alpha=16.0, scale=0.25, a_std="1/K", b_std=0.01, w_std=0.02),
    4: dict(name="gate-4096x14336-sweep-r16", projections=[("gate", 14336, 4096)], M=None, r=16,
            alpha=32.0, scale=2.0, a_std="1/K", b_std=0.01, w_std=0.02,
            M_sweep=[1, 16, 128, 1024, 8192, 32768]),
}


def layer_inputs(workload: int, projection: int, M: int | None = None):
    """(X, W, A, B, dY, scale) bf16 bit arrays for one projection of a workload."""
    w = WORKLOADS[workload]
    _, N, K = w["projections"][projection]
    M = w["M"] if M is None else M
    r = w["r"]
    X = gaussian_bf16((M, K), 1.0, seed_for(workload, "X", projection))
    W = gaussian_bf16((N, K), w["w_std"], seed_for(workload, "W", projection))
    a_std = 1.0 / K if w["a_std"] == "1/K" else float(w["a_std"])
    A = gaussian_bf16((r, K), a_std, seed_for(workload, "A", projection))
    B = gaussian_bf16((N, r), w["b_std"], seed_for(workload, "B", projection))
    dY = gaussian_bf16((M, N), 1.0, seed_for(workload, "dY", projection))
    return X, W, A, B, dY, w["scale"]
