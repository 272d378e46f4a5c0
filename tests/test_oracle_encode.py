"""Pins of the oracle's first-level quantizer (blockwise absmax + nearest NF4 level).

Pages: each weight is mapped to the closest value of the NF4 table, once,
before training (ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU",
section "NF4 Quantization: Beyond Standard INT4"). Block size 64 and the
high-nibble-first packing are readings stated in the design notes.
"""
from fractions import Fraction

import numpy as np

from bit_quantized_lora_double_b300 import synth


def exact_nearest(x, L):
    """Nearest level in exact rational arithmetic, ties to the lower code."""
    fx = Fraction(float(x))
    d = [abs(fx - Fraction(float(v))) for v in L]
    best = 0
    for i in range(1, 16):
        if d[i] < d[best]:
            best = i
    return best


def threshold_count(x, L):
    """Second formulation: the number of exact midpoints strictly below x."""
    fx = Fraction(float(x))
    return sum(1 for i in range(15) if fx > (Fraction(float(L[i])) + Fraction(float(L[i + 1]))) / 2)


def neighbours(v, k):
    """The fp32 values within k ulps of v (v rounded to fp32 first)."""
    f = np.float32(v)
    out = [f]
    up = dn = f
    for _ in range(k):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return out


def test_nearest_near_every_midpoint(oracle):
    L = oracle.nf4_table()
    xs = []
    for i in range(15):
        m = (float(L[i]) + float(L[i + 1])) / 2
        xs += neighbours(m, 8)
    xs += [np.float32(v) for v in L]
    for x in xs:
        c = oracle.nf4_nearest(x, L)
        assert c == exact_nearest(x, L) == threshold_count(x, L), (x, c)


def test_nearest_random(oracle):
    L = oracle.nf4_table()
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.uniform(-1, 1, 20000), rng.normal(0, 0.3, 5000).clip(-1, 1)]).astype(np.float32)
    for x in xs:
        c = oracle.nf4_nearest(x, L)
        assert c == threshold_count(x, L), (x, c)


def test_exact_tie_goes_to_lower_code(oracle):
    # The NF4 midpoints are not all representable in fp32, so the tie rule is
    # checked on a table whose levels 10 and 11 are moved to 0.25 and 0.3125
    # (still increasing; their midpoint 0.28125 is exact in fp32).
    L = oracle.nf4_table()
    custom = L.copy()
    custom[10] = np.float32(0.25)
    custom[11] = np.float32(0.3125)
    assert np.all(np.diff(custom) > 0)
    assert oracle.nf4_nearest(np.float32(0.28125), custom) == 10
    assert oracle.nf4_nearest(np.nextafter(np.float32(0.28125), np.float32(1)), custom) == 11
    assert oracle.nf4_nearest(np.nextafter(np.float32(0.28125), np.float32(0)), custom) == 10


def test_roundtrip_every_level(oracle):
    # A block holding a*L[i] (a a power of two, rounded to bf16) with one element
    # equal to a quantizes back to code i, and the absmax is exactly a.
    L = oracle.nf4_table()
    for a in [2.0 ** -6, 2.0 ** -1, 1.0, 8.0]:
        vals = np.zeros(64, np.float32)
        vals[0] = a
        for i in range(16):
            vals[1 + i] = np.float32(a * float(L[i]))
            vals[17 + 2 * i] = np.float32(a * float(L[15 - i]))
        W = synth.f32_to_bf16_bits(vals).reshape(1, 64)
        codes, absmax = oracle.nf4_encode(W)
        assert absmax[0] == np.float32(a)
        nib = np.empty(64, np.int64)
        nib[0::2] = codes >> 4
        nib[1::2] = codes & 15
        assert nib[0] == 15
        for i in range(16):
            assert nib[1 + i] == i
            assert nib[17 + 2 * i] == 15 - i
            assert nib[18 + 2 * i] == 7  # the zeros between them


def test_packing_high_nibble_first(oracle):
    vals = np.zeros(64, np.float32)
    vals[0], vals[1] = 1.0, -1.0
    W = synth.f32_to_bf16_bits(vals).reshape(1, 64)
    codes, _ = oracle.nf4_encode(W)
    assert codes[0] == 0xF0
    assert np.all(codes[1:] == 0x77)


def test_zero_block_and_absmax(oracle):
    W = synth.gaussian_bf16((4, 128), 0.02, 3)
    W[1, 64:] = 0
    codes, absmax = oracle.nf4_encode(W)
    f = synth.bf16_bits_to_f32(W).reshape(-1, 64)
    assert np.array_equal(absmax, np.abs(f).max(axis=1))
    assert absmax[3] == 0 and np.all(codes[3 * 32:4 * 32] == 0x77)


def test_codes_monotone_in_weight(oracle):
    rng = np.random.default_rng(11)
    v = np.sort(rng.normal(0, 1, 64)).astype(np.float32)
    W = synth.f32_to_bf16_bits(v).reshape(1, 64)
    codes, _ = oracle.nf4_encode(W)
    nib = np.empty(64, np.int64)
    nib[0::2] = codes >> 4
    nib[1::2] = codes & 15
    assert np.all(np.diff(nib) >= 0)
    assert nib[-1] == 15 or nib[0] == 0
