"""Pins of the oracle's LoRA linear layer, forward and backward.

Pages: gradients flow through the frozen 4-bit weights into the low-rank
adapters, only the adapters train (inquiringlines.com note, mechanism
paragraph; xingyuzhitong.com "Fine-Tuning Memory Requirements", section
"QLoRA: quantize the frozen base to 4 bits"); LoRA adds r x (d_in + d_out)
parameters per matrix (same page, section "LoRA: freeze the base, train small
adapters"). The forward is Y = X W'^T + s (X A^T) B^T.

Each output is linear in each of X, A and B, so a two-point difference of
L = <dY, Y> over one input element gives that element's gradient exactly up
to rounding: this pins dX, dA and dB to the forward, with no formula retyped.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth


def f64(h):
    return synth.bf16_bits_to_f32(h).astype(np.float64)


def tiny(seed, M=3, N=5, K=64, r=2):
    X = synth.gaussian_bf16((M, K), 1.0, seed)
    W = synth.gaussian_bf16((N, K), 0.5, seed + 1)
    A = synth.gaussian_bf16((r, K), 0.5, seed + 2)
    B = synth.gaussian_bf16((N, r), 0.5, seed + 3)
    dY = synth.gaussian_bf16((M, N), 1.0, seed + 4)
    return X, W, A, B, dY


def loss(oracle, X, W, A, B, dY, s):
    Y, _ = oracle.linear_fwd(X, W, A, B, s)
    return float(np.sum(Y * f64(dY)))


def two_point(oracle, args, name, idx, s):
    X, W, A, B, dY = args
    arrs = dict(X=X, A=A, B=B)
    t = arrs[name].copy()
    v0, v1 = np.float32(-1.0), np.float32(1.5)
    out = []
    for v in (v0, v1):
        t[idx] = synth.f32_to_bf16_bits(np.array([v], np.float32))[0]
        a2 = dict(arrs)
        a2[name] = t
        out.append(loss(oracle, a2["X"], W, a2["A"], a2["B"], dY, s))
    return (out[1] - out[0]) / (float(v1) - float(v0))


@pytest.mark.parametrize("s", [2.0, 0.25])
def test_gradients_by_two_point_difference(oracle, s):
    args = tiny(100)
    X, W, A, B, dY = args
    dX, dA, dB = oracle.linear_bwd(dY, X, W, A, B, s)
    for name, g in (("X", dX), ("A", dA), ("B", dB)):
        for idx in np.ndindex(g.shape):
            fd = two_point(oracle, args, name, idx, s)
            assert abs(fd - g[idx]) <= 1e-10 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


def test_scale_zero_is_plain_matmul(oracle):
    X, W, A, B, dY = tiny(200, M=7, N=9, K=128, r=4)
    Y, _ = oracle.linear_fwd(X, W, A, B, 0.0)
    np.testing.assert_allclose(Y, f64(X) @ f64(W).T, rtol=1e-12, atol=1e-12)
    dX, dA, dB = oracle.linear_bwd(dY, X, W, A, B, 0.0)
    np.testing.assert_allclose(dX, f64(dY) @ f64(W), rtol=1e-12, atol=1e-12)
    assert np.all(dA == 0) and np.all(dB == 0)


def test_zero_weight_is_pure_lora(oracle):
    X, W, A, B, dY = tiny(300, M=6, N=8, K=192, r=3)
    W[:] = 0
    Y, U = oracle.linear_fwd(X, W, A, B, 2.0)
    np.testing.assert_allclose(U, f64(X) @ f64(A).T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(Y, 2.0 * (f64(X) @ f64(A).T) @ f64(B).T, rtol=1e-11, atol=1e-13)


def test_row_and_column_subsets(oracle):
    X, W, A, B, dY = tiny(400, M=9, N=7, K=128, r=3)
    Y, _ = oracle.linear_fwd(X, W, A, B, 0.5)
    rows = [8, 0, 3]
    Ys, _ = oracle.linear_fwd(X, W, A, B, 0.5, rows=rows)
    assert np.array_equal(Ys, Y[rows])
    dX, dA, dB = oracle.linear_bwd(dY, X, W, A, B, 0.5)
    dXs, dAs, dBs = oracle.linear_bwd(dY, X, W, A, B, 0.5, rows=rows, ncols=[6, 1], kcols=[127, 5, 64])
    assert np.array_equal(dXs, dX[rows])
    assert np.array_equal(dBs, dB[[6, 1]])
    assert np.array_equal(dAs, dA[:, [127, 5, 64]])


def test_brute_force_single_output(oracle):
    # one output element written out by hand, term by term
    X, W, A, B, dY = tiny(500, M=2, N=3, K=64, r=2)
    s = 2.0
    Y, _ = oracle.linear_fwd(X, W, A, B, s)
    x, w, a, b = f64(X), f64(W), f64(A), f64(B)
    m, n = 1, 2
    base = sum(x[m, k] * w[n, k] for k in range(64))
    u = [sum(x[m, k] * a[j, k] for k in range(64)) for j in range(2)]
    lora = sum(u[j] * b[n, j] for j in range(2))
    assert abs(Y[m, n] - (base + s * lora)) < 1e-12
