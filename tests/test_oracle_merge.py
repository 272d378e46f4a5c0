"""Pins of the oracle's adapter merge (deployment: the adapters are merged into
the base weights; xingyuzhitong.com "Fine-Tuning Memory Requirements", section
"Choosing a method").

The merged weight must reproduce the adapted layer: X merged^T equals
X W'^T + s (X A^T) B^T up to the bf16 rounding of the merged weights. The
fp32 summation order over the rank (ascending j, no fused multiply-add) is a
reading, pinned by a case where the order changes the result.
"""
import numpy as np

from bit_quantized_lora_double_b300 import synth


def f32(v):
    return synth.bf16_bits_to_f32(np.asarray(v, np.uint16)).astype(np.float64)


def test_merged_weight_reproduces_the_adapted_layer(oracle):
    # A strong adapter (A ~ N(0, 1/32)) so the LoRA term is a visible share
    N, K, r, s, M = 96, 256, 8, 2.0, 16
    W = synth.gaussian_bf16((N, K), 0.02, 41)
    A = synth.gaussian_bf16((r, K), 1.0 / 32, 42)
    B = synth.gaussian_bf16((N, r), 0.05, 43)
    X = synth.gaussian_bf16((M, K), 1.0, 44)
    Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
    merged = oracle.lora_merge(Wdq, A, B, s)
    y_merged = f32(X) @ f32(merged).T
    y_adapted, _ = oracle.linear_fwd(X, Wdq, A, B, s)
    lora = s * (f32(X) @ f32(A).T) @ f32(B).T
    assert np.linalg.norm(lora) > 0.2 * np.linalg.norm(y_adapted)  # the adapter matters here
    rel = np.linalg.norm(y_merged - y_adapted) / np.linalg.norm(y_adapted)
    # merged weights carry one bf16 rounding each (relative 2^-9 at most)
    assert rel < 4e-3, rel
    # a transposed or unscaled adapter would be far off
    wrong = f32(X) @ (f32(Wdq) + (f32(B) @ f32(A))).T
    assert np.linalg.norm(wrong - y_adapted) / np.linalg.norm(y_adapted) > 0.05


def test_zero_adapter_leaves_the_base(oracle):
    W = synth.gaussian_bf16((33, 192), 0.02, 45)
    Wdq = oracle.nf4_dequantize(oracle.nf4_quantize(W))
    A = synth.gaussian_bf16((4, 192), 0.1, 46)
    B = np.zeros((33, 4), np.uint16)
    assert np.array_equal(oracle.lora_merge(Wdq, A, B, 2.0), Wdq)


def test_one_hot_adapter_hand_values(oracle):
    # W' = 0; A picks input features 3 and 5 (A[0, 3] = 1, A[1, 5] = 0.5), so
    # merged[n, 3] = s * B[n, 0] and merged[n, 5] = s * 0.5 * B[n, 1], zero elsewhere
    N, K = 4, 64
    Wdq = np.zeros((N, K), np.uint16)
    A = np.zeros((2, K), np.uint16)
    A[0, 3] = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    A[1, 5] = synth.f32_to_bf16_bits(np.float32([0.5]))[0]
    Bv = np.float32([[0.25, -1.0], [3.0, 0.125], [-0.5, 2.0], [1.5, -0.75]])
    B = synth.f32_to_bf16_bits(Bv)
    m = f32(oracle.lora_merge(Wdq, A, B, 2.0))
    expect = np.zeros((N, K))
    expect[:, 3] = 2.0 * Bv[:, 0]
    expect[:, 5] = 2.0 * 0.5 * Bv[:, 1]
    assert np.array_equal(m, expect)


def test_rank_sum_runs_in_ascending_order(oracle):
    # products 2^24, 1, -2^24 for j = 0, 1, 2: ascending fp32 order gives
    # (2^24 + 1) - 2^24 = 0 (2^24 + 1 rounds to 2^24); a descending or exact
    # sum would give 1
    K = 64
    Wdq = np.zeros((1, K), np.uint16)
    A = np.zeros((3, K), np.uint16)
    A[:, 0] = synth.f32_to_bf16_bits(np.float32([2.0 ** 12, 1.0, -2.0 ** 12]))
    B = synth.f32_to_bf16_bits(np.float32([[2.0 ** 12, 1.0, 2.0 ** 12]]))
    assert f32(oracle.lora_merge(Wdq, A, B, 1.0))[0, 0] == 0.0


def test_merge_requantize_is_quantize_of_merged(oracle):
    W = synth.gaussian_bf16((40, 128), 0.02, 47)
    A = synth.gaussian_bf16((3, 128), 0.05, 48)
    B = synth.gaussian_bf16((40, 3), 0.05, 49)
    qw = oracle.nf4_quantize(W)
    m = oracle.lora_merge(oracle.nf4_dequantize(qw), A, B, 1.5)
    a, b = oracle.merge_requantize(qw, A, B, 1.5), oracle.nf4_quantize(m)
    for key in ("codes", "absmax_q", "absmax_scale"):
        assert np.array_equal(a[key], b[key])
