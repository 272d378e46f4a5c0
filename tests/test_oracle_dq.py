"""Pins of the oracle's double quantization and decode.

Pages: double quantization quantizes the quantization constants themselves
(inquiringlines.com note, mechanism paragraph), storing them as INT8
(ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section "Double
Quantization: Squeezing the Constants"); dequantization happens on the fly to
the bf16 compute type (same section; serverroom.net, section "What LoRA and
QLoRA change in memory"). The symmetric int8 code per block, the fp32 scale
per group of 256 blocks and the single fp32 mean are readings.
"""
import math
from fractions import Fraction

import numpy as np

from bit_quantized_lora_double_b300 import synth


def test_pairwise_tree_shape(oracle):
    big = np.float32(2.0 ** 60)
    # adjacent pairs first: (big + 1) + (-big + 1) == 0 in double
    assert oracle.pairwise_sum(np.array([big, 1, -big, 1], np.float32)) == 0.0
    # a sequential sum would give 1 here, the exact sum 2
    assert math.fsum([2.0 ** 60, 1, -2.0 ** 60, 1]) == 2.0
    # padding with zeros to a power of two: (big + -big) + (1 + 0) == 1
    assert oracle.pairwise_sum(np.array([big, -big, 1], np.float32)) == 1.0
    assert oracle.pairwise_sum(np.array([], np.float32)) == 0.0


def test_pairwise_exact_when_representable(oracle):
    rng = np.random.default_rng(5)
    v = (rng.integers(1, 2 ** 16, 10007) / 2.0 ** 18).astype(np.float32)  # dyadic, exact sums
    assert oracle.pairwise_sum(v) == math.fsum(float(x) for x in v)


def test_mean_is_rounded_average(oracle):
    rng = np.random.default_rng(6)
    a = (rng.integers(1, 2 ** 12, 3000) / 2.0 ** 14).astype(np.float32)
    _, _, mean = oracle.dq_encode(a)
    exact = Fraction(math.fsum(float(x) for x in a)) / len(a)
    # mean = fp32(fp64(S / nb)): within half an fp32 ulp (plus the fp64 step)
    err = abs(Fraction(float(mean)) - exact)
    ulp = Fraction(float(np.spacing(np.float32(mean))))
    assert err <= ulp / 2 * Fraction(1000001, 1000000)


def test_constant_absmax_reduces_to_mean(oracle):
    a = np.full(1000, np.float32(0.0732421875), np.float32)
    q, s, mean = oracle.dq_encode(a)
    assert mean == a[0]
    assert np.all(s == 0) and np.all(q == 0)
    assert oracle.dq_decode(0, 0.0, mean) == a[0]


def test_group_extreme_maps_to_127(oracle):
    W = synth.gaussian_bf16((64, 4096), 0.02, 9)
    qw = oracle.nf4_quantize(W)
    q, s = qw["absmax_q"], qw["absmax_scale"]
    nb = q.size
    assert s.size == (nb + 255) // 256
    assert q.min() >= -127 and q.max() <= 127
    for g in range(s.size):
        qg = q[g * 256:(g + 1) * 256].astype(np.int64)
        if s[g] > 0:
            assert np.abs(qg).max() == 127


def test_reconstruction_error_bound(oracle):
    W = synth.gaussian_bf16((96, 4096 + 64 * 37), 0.02, 10)  # partial last group
    qw = oracle.nf4_quantize(W)
    a = qw["absmax_exact"].astype(np.float64)
    q, s, mean = qw["absmax_q"], qw["absmax_scale"], qw["absmax_mean"]
    for b in range(0, a.size, 7):
        s2 = float(s[b // 256])
        ap = float(oracle.dq_decode(q[b], s2, mean))
        tol = s2 / 2 + 4 * float(np.spacing(np.float32(max(abs(ap), abs(a[b]), 1e-30))))
        assert abs(ap - a[b]) <= tol, (b, ap, a[b], s2)


def test_storage_saving_formula():
    # bits per parameter of the constants: fp32 absmax per 64 weights, versus an
    # 8-bit code per 64 weights plus one fp32 scale per 256 blocks.
    plain = Fraction(32, 64)
    dq = Fraction(8, 64) + Fraction(32, 64 * 256)
    assert float(plain - dq) == 0.373046875


def test_dequant_roundtrip_exact(oracle):
    # All blocks share absmax a (a power of two) -> the double quantization is
    # exact (s2 = 0, a' = mean = a) and every weight of the form bf16(a * L[i])
    # decodes back to itself: codes, nibble order, levels and a' are all pinned.
    L = oracle.nf4_table()
    a = 0.0625
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 16, size=(8, 256))
    codes[:, ::64] = 15  # one +a per block fixes the absmax
    vals = (a * L.astype(np.float64)[codes]).astype(np.float32)
    W = synth.f32_to_bf16_bits(vals)
    qw = oracle.nf4_quantize(W)
    assert np.all(qw["absmax_scale"] == 0) and qw["absmax_mean"] == np.float32(a)
    Wd = oracle.nf4_dequantize(qw)
    assert np.array_equal(Wd, W)


def test_dequant_error_gaussian(oracle):
    W = synth.gaussian_bf16((128, 1024), 0.02, 13)
    qw = oracle.nf4_quantize(W)
    Wd = oracle.nf4_dequantize(qw)
    w = synth.bf16_bits_to_f32(W).astype(np.float64)
    wd = synth.bf16_bits_to_f32(Wd).astype(np.float64)
    rel = np.linalg.norm(w - wd) / np.linalg.norm(w)
    # 16 levels on Gaussian blocks: relative RMS error around 0.1 (and not zero)
    assert 0.03 < rel < 0.15, rel
    # the largest gap between levels bounds the per-weight error (plus DQ error)
    L = oracle.nf4_table().astype(np.float64)
    a = qw["absmax_exact"].astype(np.float64).repeat(64).reshape(W.shape)
    gap = np.max(np.diff(L)) / 2
    assert np.all(np.abs(w - wd) <= a * (gap + 0.02) + 1e-6)


def test_zero_block_decodes_to_zero(oracle):
    W = synth.gaussian_bf16((2, 512), 0.02, 14)
    W[0, :64] = 0
    qw = oracle.nf4_quantize(W)
    Wd = oracle.nf4_dequantize(qw)
    assert np.all(synth.bf16_bits_to_f32(Wd[0, :64]) == 0)


def _tie_absmax():
    """Absmax values whose int8 step lands exactly half-way between codes.

    With s2 = 2^-10 and mean = s2 / 2, group 0 holds c / s2 = 127 (which fixes
    s2 exactly), 2.5, 0.5, 1.5, 3.5 and -0.5; group 1 only balances the sum so
    that the mean is exactly s2 / 2. Every value is a small dyadic number, so
    the pairwise sum, the mean, c and c / s2 are all exact, and every absmax
    is a bf16 number (at most 8 significant bits), so a weight block can carry
    it.
    """
    s2 = 2.0 ** -10
    c0 = [127.0, 2.5, 0.5, 1.5, 3.5] + [-0.5] * 251      # sum 9.5
    c1 = [-0.5] * 19 + [0.0] * 237                       # sum -9.5
    a = (np.array(c0 + c1) + 0.5) * s2
    return a.astype(np.float32), s2


def test_dq_half_way_ties_round_to_even(oracle):
    # The int8 step rounds half to even (C rint): 2.5 -> 2, 0.5 -> 0,
    # -0.5 -> 0, 1.5 -> 2, 3.5 -> 4. Rounding half away from zero would give
    # 3, 1, -1 for the first three, so a round() in place of rint() fails here.
    a, s2 = _tie_absmax()
    q, s, mean = oracle.dq_encode(a)
    assert mean == np.float32(s2 / 2)
    assert s[0] == np.float32(s2)
    assert list(q[:6]) == [127, 2, 0, 2, 4, 0]
    assert np.all(q[6:256] == 0)
    # decode: a' = q * s2 + mean, exact here
    assert oracle.dq_decode(2, s2, mean) == np.float32(2.5 * s2)
