"""Python face of the CPU oracle (test infrastructure only).

The arithmetic lives in ``qlora_oracle.c``; this module builds it with gcc on
first use, loads it with ctypes and converts numpy arrays. Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import this module; the
GPU library never does.

bf16 tensors travel as numpy ``uint16`` arrays holding the bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlora_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
             "-Wall", "-Wextra", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compiles the oracle into ``oracle/liboracle.so`` (plain gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, vp, f32, f64, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_double, ctypes.c_int
            L.oracle_set_threads.restype = None
            L.oracle_set_threads.argtypes = [i32]
            L.oracle_max_threads.restype = i32
            L.oracle_max_threads.argtypes = []
            L.oracle_norm_ppf.restype = f64
            L.oracle_norm_ppf.argtypes = [f64]
            L.oracle_norm_cdf.restype = f64
            L.oracle_norm_cdf.argtypes = [f64]
            L.oracle_nf4_delta.restype = f64
            L.oracle_nf4_prob.restype = f64
            L.oracle_nf4_prob.argtypes = [i32, i32]
            L.oracle_nf4_table.argtypes = [vp]
            L.oracle_nf4_nearest.restype = i32
            L.oracle_nf4_nearest.argtypes = [f32, vp]
            L.oracle_f32_to_bf16.restype = ctypes.c_uint16
            L.oracle_f32_to_bf16.argtypes = [f32]
            L.oracle_nf4_encode.argtypes = [vp, i64, vp, vp]
            L.oracle_pairwise_sum.restype = f64
            L.oracle_pairwise_sum.argtypes = [vp, i64]
            L.oracle_dq_encode.argtypes = [vp, i64, vp, vp, vp]
            L.oracle_nf4_quantize.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp]
            L.oracle_dq_decode.restype = f32
            L.oracle_dq_decode.argtypes = [ctypes.c_int8, f32, f32]
            L.oracle_nf4_dequantize.argtypes = [vp, vp, vp, f32, i64, i64, vp]
            L.oracle_lora_down.argtypes = [vp, i64, i64, vp, i32, vp]
            L.oracle_lora_up_t.argtypes = [vp, i64, i64, vp, i32, vp]
            L.oracle_linear_fwd.argtypes = [vp, i64, vp, i64, i64, vp, vp, i32, f32, vp, i64, vp, vp]
            L.oracle_linear_bwd.argtypes = [vp, vp, i64, vp, i64, i64, vp, vp, i32, f32,
                                            vp, i64, vp, i64, vp, i64, vp, vp, vp]
            L.oracle_lora_merge.argtypes = [vp, i64, i64, vp, vp, i32, f32, vp]
            L.oracle_adamw_step.argtypes = [vp, vp, vp, vp, i64, f64, f64, f64, f64, f64, i64]
            L.oracle_int4_table.argtypes = [vp]
            L.oracle_q4_encode.argtypes = [vp, i64, vp, vp, vp]
            L.oracle_q4_dequantize_dq.argtypes = [vp, vp, vp, f32, i64, i64, vp, vp]
            L.oracle_q4_dequantize_f32.argtypes = [vp, vp, i64, i64, vp, vp]
            _lib = L
    return _lib


# -------------------------------------------------------------- threads ----

def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle's loops use from now on."""
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ---------------------------------------------------------------- table ----

def nf4_table() -> np.ndarray:
    """The 16 fp32 NF4 levels (ascending; code 7 is 0)."""
    L = np.zeros(16, np.float32)
    lib().oracle_nf4_table(_p(L))
    return L


def nf4_nearest(x: float, table: np.ndarray | None = None) -> int:
    t = nf4_table() if table is None else np.ascontiguousarray(table, np.float32)
    return int(lib().oracle_nf4_nearest(ctypes.c_float(float(np.float32(x))), _p(t)))


def norm_ppf(p: float) -> float:
    return float(lib().oracle_norm_ppf(p))


def norm_cdf(x: float) -> float:
    return float(lib().oracle_norm_cdf(x))


def nf4_prob(j: int, n: int) -> float:
    return float(lib().oracle_nf4_prob(j, n))


def nf4_delta() -> float:
    return float(lib().oracle_nf4_delta())


# ---------------------------------------------------------------- codec ----

def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def nf4_encode(W: np.ndarray):
    """First level only: (packed codes uint8[n/2], exact absmax float32[n/64])."""
    W = _u16(W)
    n = W.size
    assert n % 64 == 0
    codes = np.zeros(n // 2, np.uint8)
    absmax = np.zeros(n // 64, np.float32)
    lib().oracle_nf4_encode(_p(W), n, _p(codes), _p(absmax))
    return codes, absmax


def pairwise_sum(v: np.ndarray) -> float:
    v = np.ascontiguousarray(v, np.float32)
    return float(lib().oracle_pairwise_sum(_p(v), v.size))


def dq_encode(absmax: np.ndarray):
    """Second level: (q int8[nb], scale float32[ceil(nb/256)], mean float32)."""
    a = np.ascontiguousarray(absmax, np.float32)
    nb = a.size
    q = np.zeros(nb, np.int8)
    s = np.zeros((nb + 255) // 256, np.float32)
    mean = np.zeros(1, np.float32)
    lib().oracle_dq_encode(_p(a), nb, _p(q), _p(s), _p(mean))
    return q, s, mean[0]


def dq_decode(q: int, s2: float, mean: float) -> np.float32:
    return np.float32(lib().oracle_dq_decode(int(q), float(np.float32(s2)), float(np.float32(mean))))


def nf4_quantize(W: np.ndarray):
    """bf16 [rows, cols] -> dict(codes, absmax_q, absmax_scale, absmax_mean, absmax_exact)."""
    W = _u16(W)
    rows, cols = W.shape
    assert cols % 64 == 0
    n = rows * cols
    nb = n // 64
    codes = np.zeros(n // 2, np.uint8)
    q = np.zeros(nb, np.int8)
    s = np.zeros((nb + 255) // 256, np.float32)
    mean = np.zeros(1, np.float32)
    a = np.zeros(nb, np.float32)
    lib().oracle_nf4_quantize(_p(W), rows, cols, _p(codes), _p(q), _p(s), _p(mean), _p(a))
    return dict(codes=codes, absmax_q=q, absmax_scale=s, absmax_mean=np.float32(mean[0]),
                absmax_exact=a, rows=rows, cols=cols)


def nf4_dequantize(qw: dict) -> np.ndarray:
    """Packed weight dict -> bf16 bits uint16 [rows, cols]."""
    rows, cols = qw["rows"], qw["cols"]
    out = np.zeros((rows, cols), np.uint16)
    codes = np.ascontiguousarray(qw["codes"], np.uint8)
    q = np.ascontiguousarray(qw["absmax_q"], np.int8)
    s = np.ascontiguousarray(qw["absmax_scale"], np.float32)
    lib().oracle_nf4_dequantize(_p(codes), _p(q), _p(s), ctypes.c_float(float(qw["absmax_mean"])),
                                rows, cols, _p(out))
    return out


# --------------------------------------------------------------- linear ----

def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(rows, np.int64)
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < M))
    return r, r.size


def lora_down(X, A):
    X, A = _u16(X), _u16(A)
    M, K = X.shape
    r = A.shape[0]
    U = np.zeros((M, r), np.float64)
    lib().oracle_lora_down(_p(X), M, K, _p(A), r, _p(U))
    return U


def lora_up_t(dY, B):
    dY, B = _u16(dY), _u16(B)
    M, N = dY.shape
    r = B.shape[1]
    V = np.zeros((M, r), np.float64)
    lib().oracle_lora_up_t(_p(dY), M, N, _p(B), r, _p(V))
    return V


def linear_fwd(X, Wdq, A, B, scale, rows=None):
    """Y (fp64) for the listed rows of X (all rows if None), and U = X A^T (fp64, all rows)."""
    X, Wdq, A, B = _u16(X), _u16(Wdq), _u16(A), _u16(B)
    M, K = X.shape
    N = Wdq.shape[0]
    r = A.shape[0]
    assert Wdq.shape == (N, K) and A.shape == (r, K) and B.shape == (N, r)
    ri, nr = _rows(rows, M)
    Y = np.zeros((nr, N), np.float64)
    U = np.zeros((M, r), np.float64)
    lib().oracle_linear_fwd(_p(X), M, _p(Wdq), N, K, _p(A), _p(B), r, ctypes.c_float(scale),
                            None if ri is None else _p(ri), nr, _p(Y), _p(U))
    return Y, U


def linear_bwd(dY, X, Wdq, A, B, scale, rows=None, ncols=None, kcols=None):
    """(dX rows, dA [r, kcols], dB [ncols, r]) in fp64; None lists mean all."""
    dY, X, Wdq, A, B = _u16(dY), _u16(X), _u16(Wdq), _u16(A), _u16(B)
    M, K = X.shape
    N = Wdq.shape[0]
    r = A.shape[0]
    assert dY.shape == (M, N) and Wdq.shape == (N, K) and A.shape == (r, K) and B.shape == (N, r)
    ri, nr = _rows(rows, M)
    ni, nn = _rows(ncols, N)
    ki, nk = _rows(kcols, K)
    dX = np.zeros((nr, K), np.float64)
    dA = np.zeros((r, nk), np.float64)
    dB = np.zeros((nn, r), np.float64)
    lib().oracle_linear_bwd(_p(dY), _p(X), M, _p(Wdq), N, K, _p(A), _p(B), r, ctypes.c_float(scale),
                            None if ri is None else _p(ri), nr,
                            None if ni is None else _p(ni), nn,
                            None if ki is None else _p(ki), nk,
                            _p(dX), _p(dA), _p(dB))
    return dX, dA, dB


# --------------------------------------------------------------- groups ----
# Several LoRA linears reading the same X (q/k/v, gate/up: xingyuzhitong.com
# "Fine-Tuning Memory Requirements", section "LoRA: freeze the base, train
# small adapters"). Each output is its own projection's; the gradient of the
# shared input is the sum of the projections' (the chain rule through a value
# used n times).

def group_fwd(X, Wdqs, As, Bs, scale, rows=None):
    """[(Y_g, U_g)] for every projection g, as linear_fwd computes them."""
    return [linear_fwd(X, W, A, B, scale, rows=rows) for W, A, B in zip(Wdqs, As, Bs)]


def group_bwd(dYs, X, Wdqs, As, Bs, scale, rows=None):
    """(dX = sum over g of linear_bwd's dX_g, in fp64 in projection order, and
    [(dA_g, dB_g)])."""
    dX = None
    grads = []
    for dY, W, A, B in zip(dYs, Wdqs, As, Bs):
        dXg, dA, dB = linear_bwd(dY, X, W, A, B, scale, rows=rows)
        dX = dXg if dX is None else dX + dXg
        grads.append((dA, dB))
    return dX, grads


# ---------------------------------------------------------------- merge ----

def lora_merge(Wdq, A, B, scale):
    """bf16 merged weight W' + s * B A (fixed fp32 order, see the C source)."""
    Wdq, A, B = _u16(Wdq), _u16(A), _u16(B)
    N, K = Wdq.shape
    r = A.shape[0]
    assert A.shape == (r, K) and B.shape == (N, r)
    out = np.zeros((N, K), np.uint16)
    lib().oracle_lora_merge(_p(Wdq), N, K, _p(A), _p(B), r, ctypes.c_float(scale), _p(out))
    return out


def merge_requantize(qw: dict, A, B, scale):
    """The quantized weight of the merged layer: quantize(merge(dequant(qw)))."""
    return nf4_quantize(lora_merge(nf4_dequantize(qw), A, B, scale))


# ---------------------------------------------------------------- adamw ----

def adamw_step(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW step in fp64, in place on p, m, v (float64 arrays)."""
    for a in (p, m, v):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    g = np.ascontiguousarray(g, np.float64)
    lib().oracle_adamw_step(_p(p), _p(g), _p(m), _p(v), p.size, lr, beta1, beta2, eps, weight_decay, step)


# ------------------------------------------------------------- variants ----
# Storage variants of the 4-bit weight: the NF4 or the INT4 table, and the
# absmax double-quantized (q, scale, mean) or kept as fp32 per block.

def int4_table() -> np.ndarray:
    L = np.zeros(16, np.float32)
    lib().oracle_int4_table(_p(L))
    return L


def q4_table(table: str) -> np.ndarray:
    return nf4_table() if table == "nf4" else int4_table()


def q4_quantize(W: np.ndarray, table: str = "nf4", double_quant: bool = True):
    """bf16 [rows, cols] -> dict(codes, table, double_quant, absmax (fp32) or absmax_q/scale/mean)."""
    W = _u16(W)
    rows, cols = W.shape
    n = rows * cols
    nb = n // 64
    codes = np.zeros(n // 2, np.uint8)
    a = np.zeros(nb, np.float32)
    L = q4_table(table)
    lib().oracle_q4_encode(_p(W), n, _p(L), _p(codes), _p(a))
    out = dict(codes=codes, rows=rows, cols=cols, table=table, double_quant=double_quant, absmax_exact=a)
    if double_quant:
        q, s, mean = dq_encode(a)
        out.update(absmax_q=q, absmax_scale=s, absmax_mean=np.float32(mean))
    else:
        out.update(absmax=a.copy())
    return out


def q4_dequantize(qw: dict) -> np.ndarray:
    rows, cols = qw["rows"], qw["cols"]
    out = np.zeros((rows, cols), np.uint16)
    codes = np.ascontiguousarray(qw["codes"], np.uint8)
    L = q4_table(qw["table"])
    if qw["double_quant"]:
        q = np.ascontiguousarray(qw["absmax_q"], np.int8)
        s = np.ascontiguousarray(qw["absmax_scale"], np.float32)
        lib().oracle_q4_dequantize_dq(_p(codes), _p(q), _p(s), ctypes.c_float(float(qw["absmax_mean"])),
                                      rows, cols, _p(L), _p(out))
    else:
        a = np.ascontiguousarray(qw["absmax"], np.float32)
        lib().oracle_q4_dequantize_f32(_p(codes), _p(a), rows, cols, _p(L), _p(out))
    return out
