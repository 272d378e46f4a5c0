"""GPU codec parity: NF4 codes, int8 absmax codes, second-level scales, the
mean and the dequantized bf16 weights must equal the oracle's bit for bit."""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth

pytestmark = pytest.mark.gpu

SHAPES = [(1, 64), (3, 128), (5, 64 * 7), (64, 4096 + 64 * 37), (257, 1024), (1000, 192)]


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


def assert_quant_equal(w, qw):
    assert np.array_equal(w.codes.cpu().numpy(), qw["codes"]), "NF4 codes differ"
    assert np.array_equal(w.absmax_q.cpu().numpy(), qw["absmax_q"]), "int8 absmax codes differ"
    assert np.array_equal(w.absmax_scale.cpu().numpy().view(np.uint32), qw["absmax_scale"].view(np.uint32)), \
        "second-level scales differ"
    assert np.float32(w.absmax_mean[0].item()).view(np.uint32) == np.float32(qw["absmax_mean"]).view(np.uint32), \
        "mean differs"


@pytest.mark.parametrize("shape", SHAPES)
def test_quantize_bit_exact(g, oracle, shape):
    W = synth.gaussian_bf16(shape, 0.02, 1000 + shape[0])
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert_quant_equal(w, qw)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_decode_alone_bit_exact(g, oracle):
    W = synth.gaussian_bf16((128, 2048), 0.05, 77)
    qw = oracle.nf4_quantize(W)
    w = g.weight_from_oracle(qw)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_zero_and_constant_blocks(g, oracle):
    W = synth.gaussian_bf16((16, 512), 0.02, 5)
    W[0] = 0                     # whole zero rows: absmax 0, all codes 7
    W[3, 64:128] = 0
    W[5, :] = synth.f32_to_bf16_bits(np.full(512, 0.25, np.float32))
    qw = oracle.nf4_quantize(W)
    w = g.quantize(W)
    assert_quant_equal(w, qw)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_all_zero_weight(g, oracle):
    W = np.zeros((8, 256), np.uint16)
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert_quant_equal(w, qw)
    assert np.all(w.codes.cpu().numpy() == 0x77)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_wide_dynamic_range(g, oracle):
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((32, 1024)) * np.exp(rng.uniform(-60, 60, (32, 1)))).astype(np.float32)
    W = synth.f32_to_bf16_bits(v)
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert_quant_equal(w, qw)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_codec_full_size(g, oracle):
    # the standalone codec workload: 14336 x 4096, N(0, 0.02)
    W = synth.gaussian_bf16((14336, 4096), 0.02, synth.seed_for(2, "W"))
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert_quant_equal(w, qw)
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))


def test_dq_half_way_ties(g, oracle):
    # Blocks whose absmax puts c / s2 exactly half-way between int8 codes
    # (2.5, 0.5, -0.5 ...): the GPU's int8 step must round half to even as
    # the oracle does. Block b holds its absmax once and zeros elsewhere.
    from tests.test_oracle_dq import _tie_absmax
    a, _ = _tie_absmax()
    W = np.zeros((a.size, 64), np.uint16)
    W[:, 0] = synth.f32_to_bf16_bits(a)
    assert np.array_equal(synth.bf16_bits_to_f32(W[:, 0]), a)  # the absmax values are bf16 numbers
    W = W.reshape(8, -1)
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert_quant_equal(w, qw)
    assert list(w.absmax_q.cpu().numpy()[:6]) == [127, 2, 0, 2, 4, 0]
    assert np.array_equal(g.dequantize(w), oracle.nf4_dequantize(qw))
