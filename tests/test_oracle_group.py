"""Pins of the oracle's projection groups (several LoRA linears on one X).

A group of n projections is one LoRA linear over the stacked weight
W = [W_0; ...; W_{n-1}] with the stacked down-projection A = [A_0; ...] and a
block-diagonal up-projection (B_g in rows of projection g, columns
[g r, (g + 1) r)): Y = X W^T + s (X A^T) B^T is [Y_0 ... Y_{n-1}] side by
side, and the gradient of X for dY = [dY_0 ... dY_{n-1}] is the group's dX.
The single-layer oracle computes that stacked layer independently of the
group functions, so the two agree up to fp64 rounding; a dropped projection,
a wrong pairing of dY_g with W_g or B_g, or a wrong sign in the sum fails.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth


def make(seed, M, Ns, K, r):
    X = synth.gaussian_bf16((M, K), 1.0, seed)
    Ws = [synth.gaussian_bf16((N, K), 0.5, seed + 10 * g + 1) for g, N in enumerate(Ns)]
    As = [synth.gaussian_bf16((r, K), 0.5, seed + 10 * g + 2) for g in range(len(Ns))]
    Bs = [synth.gaussian_bf16((N, r), 0.5, seed + 10 * g + 3) for g, N in enumerate(Ns)]
    dYs = [synth.gaussian_bf16((M, N), 1.0, seed + 10 * g + 4) for g, N in enumerate(Ns)]
    return X, Ws, As, Bs, dYs


def stacked(Ws, As, Bs, dYs, r):
    n = len(Ws)
    W = np.vstack(Ws)
    A = np.vstack(As)
    Bbd = np.zeros((W.shape[0], n * r), np.uint16)  # bf16 zeros
    row = 0
    for g, B in enumerate(Bs):
        Bbd[row:row + B.shape[0], g * r:(g + 1) * r] = B
        row += B.shape[0]
    return W, A, Bbd, np.hstack(dYs)


@pytest.mark.parametrize("Ns,r", [([5, 3, 3], 2), ([7, 7], 3), ([4], 1)])
def test_group_is_the_stacked_layer(oracle, Ns, r):
    M, K, s = 4, 128, 0.75
    X, Ws, As, Bs, dYs = make(7, M, Ns, K, r)
    W, A, Bbd, dY = stacked(Ws, As, Bs, dYs, r)
    outs = oracle.group_fwd(X, Ws, As, Bs, s)
    Y, U = oracle.linear_fwd(X, W, A, Bbd, s)
    assert np.allclose(np.hstack([y for y, _ in outs]), Y, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.hstack([u for _, u in outs]), U, rtol=1e-12, atol=1e-12)
    dX, grads = oracle.group_bwd(dYs, X, Ws, As, Bs, s)
    dXs, dAs, dBs = oracle.linear_bwd(dY, X, W, A, Bbd, s)
    assert np.allclose(dX, dXs, rtol=1e-12, atol=1e-12)
    # dA of the stacked layer is the projections' dA stacked; dB its blocks
    assert np.allclose(np.vstack([a for a, _ in grads]), dAs, rtol=1e-12, atol=1e-12)
    row = 0
    for g, (_, dB) in enumerate(grads):
        n = dB.shape[0]
        assert np.allclose(dB, dBs[row:row + n, g * r:(g + 1) * r], rtol=1e-12, atol=1e-12)
        row += n


def test_group_rows_subset(oracle):
    X, Ws, As, Bs, dYs = make(3, 9, [6, 2], 64, 2)
    full, _ = oracle.group_bwd(dYs, X, Ws, As, Bs, 1.5)
    rows = np.array([0, 4, 8])
    sub, _ = oracle.group_bwd(dYs, X, Ws, As, Bs, 1.5, rows=rows)
    assert np.array_equal(sub, full[rows])
