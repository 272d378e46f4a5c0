"""GPU parity of the storage variants: the INT4 level table (16 evenly spaced
levels, the baseline NF4 is compared against) and the block absmax kept in
fp32 without double quantization, each alone and together, through every
kernel: quantize and dequantize bit for bit against the oracle, the linear
forward (few-token, small-M and tensor-core paths) and backward (CUDA-core and
tensor-core paths) within the linear layer's bar (relative Frobenius error
<= 5e-3, the same arithmetic argument as for NF4 with double quantization).

Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
"NF4 Quantization: Beyond Standard INT4"; xingyuzhitong.com "Fine-Tuning
Memory Requirements", section "QLoRA: quantize the frozen base to 4 bits"
(4.5 bits per weight with one fp32 constant per 64 weights).
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth

pytestmark = pytest.mark.gpu
TOL = 5e-3
FORMATS = [("nf4", True), ("nf4", False), ("int4", True), ("int4", False)]


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


def _check_weight(g, w, qw):
    assert np.array_equal(w.codes.cpu().numpy(), qw["codes"]), "codes"
    if qw["double_quant"]:
        assert np.array_equal(w.absmax_q.cpu().numpy(), qw["absmax_q"]), "absmax codes"
        assert np.array_equal(w.absmax_scale.cpu().numpy().view(np.uint32), qw["absmax_scale"].view(np.uint32))
        assert np.float32(w.absmax_mean[0].item()).view(np.uint32) == np.float32(qw["absmax_mean"]).view(np.uint32)
    else:
        nb = len(qw["absmax"])
        assert np.array_equal(w.absmax[:nb].cpu().numpy().view(np.uint32), qw["absmax"].view(np.uint32))


@pytest.mark.parametrize("table,dq", FORMATS)
@pytest.mark.parametrize("rows,cols,seed", [
    (300, 1024, 1),    # 4800 blocks: 18 full second-level groups and a ragged one
    (1, 64, 2),        # one block
    (97, 4096, 3),     # several groups, odd row count
])
def test_quantize_dequantize_bit_exact(g, oracle, table, dq, rows, cols, seed):
    W = synth.gaussian_bf16((rows, cols), 0.02, seed)
    qw = oracle.q4_quantize(W, table, dq)
    w = g.q4_quantize(W, table, dq)
    _check_weight(g, w, qw)
    assert np.array_equal(g.dequantize(w), oracle.q4_dequantize(qw))


@pytest.mark.parametrize("table,dq", FORMATS)
def test_quantize_degenerate_blocks(g, oracle, table, dq):
    # all-zero blocks (absmax 0: every code the exact zero), one-hot blocks,
    # and blocks whose entries sit exactly on the table's levels
    rows, cols = 8, 256
    W = synth.gaussian_bf16((rows, cols), 0.02, 9)
    W[0, :] = 0
    W[1, :] = 0
    W[1, 5] = synth.f32_to_bf16_bits(np.array([-0.75], np.float32))[0]
    L = oracle.q4_table(table)
    lv = synth.f32_to_bf16_bits((L[:15] if table == "int4" else L).astype(np.float32))
    W[2, :len(lv)] = lv
    qw = oracle.q4_quantize(W, table, dq)
    w = g.q4_quantize(W, table, dq)
    _check_weight(g, w, qw)
    assert np.array_equal(g.dequantize(w), oracle.q4_dequantize(qw))


@pytest.mark.parametrize("table,dq", FORMATS)
def test_dequantize_from_oracle_weights(g, oracle, table, dq):
    W = synth.gaussian_bf16((200, 2048), 0.05, 21)
    qw = oracle.q4_quantize(W, table, dq)
    w = g.q4_weight_from_oracle(qw)
    assert np.array_equal(g.dequantize(w), oracle.q4_dequantize(qw))


def _linear(g, oracle, table, dq, M, N, K, r, scale, seed, bwd=True):
    X = synth.gaussian_bf16((M, K), 1.0, seed)
    W = synth.gaussian_bf16((N, K), 0.02, seed + 1)
    A = synth.gaussian_bf16((r, K), 1.0 / K, seed + 2)
    B = synth.gaussian_bf16((N, r), 0.01, seed + 3)
    dY = synth.gaussian_bf16((M, N), 1.0, seed + 4)
    qw = oracle.q4_quantize(W, table, dq)
    Wdq = oracle.q4_dequantize(qw)
    w = g.q4_weight_from_oracle(qw)
    Y, U = g.fwd(X, w, A, B, r, scale)
    Yref, Uref = oracle.linear_fwd(X, Wdq, A, B, scale)
    errs = {"Y": g.rel_fro(g.host_f64_bf16(Y), Yref), "U": g.rel_fro(g.host_f64_bf16(U), Uref)}
    if bwd:
        dX, dA, dB = g.bwd(dY, X, U, w, A, B, r, scale)
        dXr, dAr, dBr = oracle.linear_bwd(dY, X, Wdq, A, B, scale)
        errs["dX"] = g.rel_fro(g.host_f64_bf16(dX), dXr)
        errs["dA"] = g.rel_fro(dA.cpu().numpy(), dAr)
        errs["dB"] = g.rel_fro(dB.cpu().numpy(), dBr)
    for k, v in errs.items():
        assert v <= TOL, (k, v, errs)


@pytest.mark.parametrize("table,dq", FORMATS)
@pytest.mark.parametrize("M,N,K,r,scale", [
    (5, 1000, 2048, 8, 2.0),      # few-token kernel, one 8-token tile; CUDA-core backward
    (13, 520, 1024, 16, 1.0),     # few-token kernel, two tiles
    (24, 300, 320, 5, 2.0),       # small-M kernel (M > 16, K not a multiple of 256)
    (200, 384, 512, 16, 2.0),     # tensor-core GEMM forward and backward
])
def test_linear_parity(g, oracle, table, dq, M, N, K, r, scale):
    _linear(g, oracle, table, dq, M, N, K, r, scale, seed=100 + M)


@pytest.mark.parametrize("table,dq", [("int4", False)])
def test_linear_quantized_on_device(g, oracle, table, dq):
    # the whole chain on the device: quantize, then the forward reads the
    # weight the library wrote (bit-equal to the oracle's, checked above)
    M, N, K, r = 96, 256, 1024, 8
    X = synth.gaussian_bf16((M, K), 1.0, 7)
    W = synth.gaussian_bf16((N, K), 0.02, 8)
    A = synth.gaussian_bf16((r, K), 1.0 / K, 9)
    B = synth.gaussian_bf16((N, r), 0.01, 10)
    w = g.q4_quantize(W, table, dq)
    Y, U = g.fwd(X, w, A, B, r, 2.0)
    Yref, _ = oracle.linear_fwd(X, oracle.q4_dequantize(oracle.q4_quantize(W, table, dq)), A, B, 2.0)
    assert g.rel_fro(g.host_f64_bf16(Y), Yref) <= TOL
