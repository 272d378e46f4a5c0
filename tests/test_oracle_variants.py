"""Pins of the oracle's storage variants of the 4-bit weight.

- INT4: the standard 4-bit baseline the pages compare NF4 against
  (ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section "NF4
  Quantization: Beyond Standard INT4": 16 evenly spaced levels). Reading:
  symmetric absmax INT4, levels (i - 7) / 7, nearest level with ties to the
  lower code (the NF4 tie rule).
- fp32 absmax without double quantization: 4.5 bits per weight
  (xingyuzhitong.com, section "QLoRA: quantize the frozen base to 4 bits":
  "4.5 to 5" bits per weight with the quantization constants).
"""
from fractions import Fraction

import numpy as np

from bit_quantized_lora_double_b300 import synth


def test_int4_table_is_uniform(oracle):
    L = oracle.int4_table().astype(np.float64)
    assert L[7] == 0 and L[0] == -1 and L[14] == 1
    assert np.allclose(np.diff(L), 1 / 7, rtol=0, atol=1e-7)
    assert np.allclose(L[:7], -L[14:7:-1])  # symmetric around the zero code


def test_int4_encode_rounds_to_sevenths_ties_down(oracle):
    # nearest multiple of 1/7 in exact rational arithmetic, ties to the lower
    # one; x on exact midpoints (2m + 1) / 14 rounded to fp32 included
    L = oracle.int4_table()
    rng = np.random.default_rng(5)
    xs = list(rng.uniform(-1, 1, 3000).astype(np.float32))
    xs += [np.float32((2 * m + 1) / 14) for m in range(-7, 7)]
    for x in xs:
        # the two table levels around x, compared in exact rational arithmetic
        fx = Fraction(float(x)) * 7
        lo = fx.numerator // fx.denominator
        d_lo = abs(Fraction(float(x)) - Fraction(float(L[lo + 7])))
        d_hi = abs(Fraction(float(x)) - Fraction(float(L[min(lo + 8, 15)])))
        k = lo if d_lo <= d_hi else lo + 1
        assert oracle.nf4_nearest(x, L) == k + 7, (x, k)


def test_nf4_reconstructs_gaussian_weights_better_than_int4(oracle):
    # NF4 is built for normally distributed weights (inquiringlines.com note:
    # "information theoretically optimal for normally distributed weights")
    W = synth.gaussian_bf16((256, 1024), 0.02, 61)
    w = synth.bf16_bits_to_f32(W).astype(np.float64)
    err = {}
    for table in ("nf4", "int4"):
        qw = oracle.q4_quantize(W, table, double_quant=False)
        wd = synth.bf16_bits_to_f32(oracle.q4_dequantize(qw)).astype(np.float64)
        err[table] = np.linalg.norm(w - wd) / np.linalg.norm(w)
    assert err["nf4"] < 0.9 * err["int4"], err


def test_fp32_absmax_round_trip_exact(oracle):
    # without double quantization a' is the exact absmax: any weight of the
    # form bf16(a_b * L[c]) with one +-a_b per block decodes to itself, for
    # every per-block a_b (here powers of two times 1, 1.5, 1.75)
    rng = np.random.default_rng(62)
    for table in ("nf4", "int4"):
        L = oracle.q4_table(table).astype(np.float64)
        codes = rng.integers(0, 15 if table == "int4" else 16, size=(16, 256))
        codes[:, ::64] = 14 if table == "int4" else 15
        a = (2.0 ** rng.integers(-8, 0, size=(16, 4))) * rng.choice([1.0, 1.5, 1.75], size=(16, 4))
        vals = (np.repeat(a, 64, axis=1) * L[codes]).astype(np.float32)
        W = synth.f32_to_bf16_bits(vals)
        qw = oracle.q4_quantize(W, table, double_quant=False)
        assert np.array_equal(qw["absmax"], a.reshape(-1).astype(np.float32))
        assert np.array_equal(oracle.q4_dequantize(qw), W)


def test_variant_storage_bits_per_weight():
    # codes 4 bits + fp32 absmax per 64 weights = 4.5 bits (the pages' "4.5 to 5")
    assert 4 + 32 / 64 == 4.5
    # double quantization: 4 + 8/64 + 32/(64*256)
    assert abs((4 + 8 / 64 + 32 / (64 * 256)) - 4.126953125) < 1e-12


def test_int4_with_double_quant_shares_the_constants(oracle):
    # the second level only sees the absmax values, which both tables share
    W = synth.gaussian_bf16((64, 512), 0.02, 63)
    a, b = oracle.q4_quantize(W, "nf4"), oracle.q4_quantize(W, "int4")
    for key in ("absmax_q", "absmax_scale"):
        assert np.array_equal(a[key], b[key])
    assert a["absmax_mean"] == b["absmax_mean"]
    ref = oracle.nf4_quantize(W)
    assert np.array_equal(a["codes"], ref["codes"])
    assert np.array_equal(oracle.q4_dequantize(a), oracle.nf4_dequantize(ref))
