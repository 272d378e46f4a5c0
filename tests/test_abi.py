"""The C-ABI library loads without a GPU, exports every declared symbol, and
rejects bad arguments on the host before launching anything."""
import ctypes
import json
import os
import re
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlora.h")
FIG = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_figures.json")))


@pytest.fixture(scope="module")
def q():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from bit_quantized_lora_double_b300 import qlora
    qlora.lib()
    return qlora


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlora_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(q):
    names = declared_functions()
    assert len(names) >= 14
    L = q.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(q.EXPORTS)


def test_table_matches_oracle(q, oracle):
    assert np.array_equal(q.qlora_nf4_table().view(np.uint32), oracle.nf4_table().view(np.uint32))


def test_q4_tables_match_oracle(q, oracle):
    assert np.array_equal(q.qlora_q4_table(q.TABLE_NF4).view(np.uint32), oracle.q4_table("nf4").view(np.uint32))
    assert np.array_equal(q.qlora_q4_table(q.TABLE_INT4).view(np.uint32), oracle.q4_table("int4").view(np.uint32))
    assert not q.qlora_q4_table(7).any()




def test_storage_bits_match_pages(q):
    # codes + int8 absmax per 64 weights + fp32 scale per 256 blocks
    rows, cols = 4096, 4096 * 4
    n = rows * cols
    assert q.qlora_nf4_codes_bytes(rows, cols) == n // 2
    assert q.qlora_nf4_absmax_count(rows, cols) == n // 64
    assert q.qlora_nf4_scale_count(rows, cols) == n // 64 // 256
    bits_dq = Fraction(8 * (q.qlora_nf4_absmax_count(rows, cols) + 4 * q.qlora_nf4_scale_count(rows, cols)), n)
    bits_plain = Fraction(32 * (n // 64), n)  # fp32 absmax per block, no double quantization
    saving = float(bits_plain - bits_dq)
    assert saving == 0.373046875
    g = FIG["dq_saving_bits_per_param"]
    assert abs(saving - g["value"]) <= g["tolerance"]
    g = FIG["dq_saving_bits_per_param_nested"]
    assert abs(saving - g["value"]) <= g["tolerance"]
    g = FIG["dq_saving_gb_65b"]
    assert abs(saving * g["params"] / 8 / 1e9 - g["value"]) <= g["tolerance"]
    g = FIG["dq_constant_memory_reduction"]
    assert abs(float(1 - bits_dq / bits_plain) - g["value"]) <= g["tolerance"]
    g = FIG["block_format_bits_per_weight"]
    assert g["low"] <= 4 + float(bits_plain) <= g["high"]
    total = q.qlora_nf4_storage_bytes(rows, cols)
    assert total * 8 / n == pytest.approx(4 + float(bits_dq), abs=1e-5)


def test_invalid_sizes_return_zero(q):
    assert q.qlora_nf4_codes_bytes(10, 100) == 0       # cols % 64
    assert q.qlora_nf4_codes_bytes(-1, 64) == 0
    assert q.qlora_nf4_quantize_workspace(4, 63) == 0
    assert q.qlora_nf4_codes_bytes(0, 64) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced


def desc(rows=64, cols=128, codes=FAKE, qq=FAKE, s=FAKE, m=FAKE):
    return q_mod().Nf4WeightDesc(rows, cols, codes, qq, s, m)


def q_mod():
    from bit_quantized_lora_double_b300 import qlora
    return qlora


def call_quant(q, W, d, ws, nbytes):
    return q.lib().qlora_nf4_quantize(ctypes.c_void_p(W), ctypes.byref(d), ctypes.c_void_p(ws), nbytes, None)


def test_quantize_rejects_on_host(q):
    need = q.qlora_nf4_quantize_workspace(64, 128)
    assert call_quant(q, FAKE, desc(), FAKE, need - 1) == 4
    assert "workspace" in q.qlora_last_error()
    assert call_quant(q, 0, desc(), FAKE, need) == 1
    assert call_quant(q, FAKE + 8, desc(), FAKE, need) == 3
    assert call_quant(q, FAKE, desc(cols=100), FAKE, need) == 2
    assert call_quant(q, FAKE, desc(codes=0), FAKE, need) == 1
    assert call_quant(q, FAKE, desc(s=FAKE + 4), FAKE, need) == 3
    assert call_quant(q, FAKE, desc(), 0, need) == 1


def q4desc(table=0, dq=0, rows=64, cols=128, codes=FAKE, qq=0, s=0, m=0, a=FAKE):
    return q_mod().Q4WeightDesc(rows, cols, table, dq, codes, qq, s, m, a)


def test_q4_quantize_rejects_on_host(q):
    L = q.lib()
    c = ctypes.c_void_p

    def call(d, ws=0, nbytes=0):
        return L.qlora_q4_quantize(c(FAKE), ctypes.byref(d), c(ws), nbytes, None)
    assert call(q4desc(table=2)) == 8
    assert call(q4desc(dq=2)) == 8
    assert call(q4desc(a=0)) == 1
    assert call(q4desc(a=FAKE + 4)) == 3
    # double-quantized: its three arrays and the workspace are required
    assert call(q4desc(dq=1, a=0)) == 1
    assert call(q4desc(dq=1, qq=FAKE, s=FAKE, m=FAKE, a=0)) == 1
    need = q.qlora_nf4_quantize_workspace(64, 128)
    assert call(q4desc(dq=1, qq=FAKE, s=FAKE, m=FAKE, a=0), FAKE, need - 1) == 4
    d = q4desc(table=1, rows=0)
    assert call(d) == 0  # no rows: nothing to launch
    assert L.qlora_q4_dequantize(ctypes.byref(q4desc(table=3)), c(FAKE), None) == 8
    assert L.qlora_q4_linear_fwd_workspace(16, ctypes.byref(q4desc()), 8) == \
        L.qlora_linear_fwd_workspace(16, ctypes.byref(desc()), 8)
    assert L.qlora_q4_linear_fwd(c(FAKE), 16, ctypes.byref(q4desc(table=9)), c(FAKE), c(FAKE), 8, 2.0, c(FAKE),
                                 None, c(FAKE), 1 << 30, None) == 8


def test_group_rejects_on_host(q):
    L = q.lib()
    c = ctypes.c_void_p
    d1, d2, d3 = desc(rows=64, cols=128), desc(rows=128, cols=128), desc(rows=64, cols=256)

    def projs(ds, **kw):
        arr = (q.ProjDesc * len(ds))()
        for i, d in enumerate(ds):
            arr[i].w = ctypes.pointer(d)
            for f in ("A", "B", "Y", "dY", "dA", "dB"):
                setattr(arr[i], f, kw.get(f, FAKE))
        return arr

    def fwd(ds, n=None, r=16, M=64, ws_bytes=1 << 40, **kw):
        return L.qlora_group_fwd(c(FAKE), M, projs(ds, **kw), len(ds) if n is None else n, r, 2.0, None, c(FAKE),
                                 ws_bytes, None)

    def bwd(ds, r=16, M=64, **kw):
        return L.qlora_group_bwd(c(FAKE), None, M, projs(ds, **kw), len(ds), r, 2.0, c(FAKE), c(FAKE), 1 << 40, None)
    assert fwd([d1, d2], n=0) == 2
    assert fwd([d1, d2], n=5) == 2
    assert fwd([d1, d2], r=12) == 5     # r % 8
    assert fwd([d1, d2], r=136) == 5
    assert fwd([d1, d3]) == 2           # different K
    assert fwd([d1, d2], A=0) == 1
    assert fwd([d1, d2], Y=0) == 1
    assert fwd([d1, d2], Y=FAKE + 8) == 3
    assert fwd([d1, d2], ws_bytes=16) == 4
    assert fwd([d1, desc(cols=100)]) == 2
    assert bwd([d1, d2], dY=0) == 1
    assert bwd([d1, d2], dA=0) == 1
    assert bwd([d1, d2], dB=FAKE + 4) == 3
    assert fwd([d1, d2], M=0) == 0      # nothing to launch
    # workspace queries: 0 for invalid groups, outputs not needed
    assert L.qlora_group_fwd_workspace(64, projs([d1, d3]), 2, 16) == 0
    assert L.qlora_group_fwd_workspace(64, projs([d1, d2], Y=0), 2, 16) > 0
    assert L.qlora_group_bwd_workspace(64, projs([d1, d2], dY=0), 2, 16) > 0
    assert L.qlora_group_bwd_workspace(64, projs([d1, d2]), 2, 12) == 0


def call_fwd(q, M=16, d=None, r=8, ws_bytes=None, X=FAKE, A=FAKE, B=FAKE, Y=FAKE):
    d = d or desc()
    if ws_bytes is None:
        ws_bytes = q.lib().qlora_linear_fwd_workspace(M, ctypes.byref(d), r)
    return q.lib().qlora_linear_fwd(ctypes.c_void_p(X), M, ctypes.byref(d), ctypes.c_void_p(A), ctypes.c_void_p(B),
                                    r, 2.0, ctypes.c_void_p(Y), None, ctypes.c_void_p(FAKE), ws_bytes, None)


def test_linear_fwd_rejects_on_host(q):
    assert call_fwd(q, r=0) == 5
    assert call_fwd(q, r=129) == 5
    assert call_fwd(q, M=-1) == 2
    assert call_fwd(q, A=0) == 1
    assert call_fwd(q, X=0) == 1
    assert call_fwd(q, Y=FAKE + 2) == 3
    assert call_fwd(q, ws_bytes=16) == 4
    assert call_fwd(q, d=desc(rows=0)) == 2
    assert call_fwd(q, d=desc(cols=96)) == 2
    # M == 0 is valid and launches nothing
    assert call_fwd(q, M=0) == 0


def test_linear_bwd_rejects_on_host(q):
    d = desc()
    L = q.lib()
    need = L.qlora_linear_bwd_workspace(16, ctypes.byref(d), 8)
    c = ctypes.c_void_p

    def call(dA=FAKE, ws_bytes=need, r=8, dY=FAKE):
        return L.qlora_linear_bwd(c(dY), c(FAKE), None, 16, ctypes.byref(d), c(FAKE), c(FAKE), r, 2.0, c(FAKE),
                                  c(dA), c(FAKE), c(FAKE), ws_bytes, None)
    assert call(dA=0) == 1
    assert call(dY=0) == 1
    assert call(ws_bytes=need - 1) == 4
    assert call(r=200) == 5
    assert call(dA=FAKE + 4) == 3


def test_workspace_queries_monotone(q):
    d = desc(rows=1024, cols=1024)
    L = q.lib()
    a = L.qlora_linear_fwd_workspace(128, ctypes.byref(d), 16)
    b = L.qlora_linear_fwd_workspace(256, ctypes.byref(d), 16)
    assert 0 < a <= b
    assert L.qlora_linear_bwd_workspace(256, ctypes.byref(d), 16) > 0
    assert L.qlora_linear_fwd_workspace(128, ctypes.byref(d), 0) == 0


def test_version(q):
    assert "sm_103a" in q.qlora_version()
