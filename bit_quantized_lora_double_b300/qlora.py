"""Thin Python binding of the C ABI in include/qlora.h (ctypes).

The functions carry the C names and only marshal arguments: tensors become
device pointers, the stream defaults to torch's current stream, a non-zero
status raises QloraError with the library's message. Every step of the
computation runs in the library's CUDA kernels. PyTorch supplies device
memory and streams.

The library must be built first (``python -m bit_quantized_lora_double_b300._build``
or ``__graft_entry__.build()``); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqlora_b300.so")
_lib = None

STATUS = {0: "QLORA_OK", 1: "QLORA_ERR_NULL", 2: "QLORA_ERR_SHAPE", 3: "QLORA_ERR_ALIGN",
          4: "QLORA_ERR_WORKSPACE", 5: "QLORA_ERR_RANK", 6: "QLORA_ERR_CUDA", 7: "QLORA_ERR_TIMEOUT",
          8: "QLORA_ERR_UNSUPPORTED"}

EXPORTS = [
    "qlora_nf4_codes_bytes", "qlora_nf4_absmax_count", "qlora_nf4_scale_count", "qlora_nf4_storage_bytes",
    "qlora_nf4_quantize_workspace", "qlora_nf4_table", "qlora_nf4_quantize", "qlora_nf4_quantize_noalloc",
    "qlora_nf4_dequantize",
    "qlora_linear_fwd_workspace", "qlora_linear_bwd_workspace", "qlora_linear_fwd", "qlora_linear_bwd",
    "qlora_last_error", "qlora_check_device_status", "qlora_set_wait_limit", "qlora_version",
    "qlora_profile_start", "qlora_profile_stop", "qlora_debug_gemm_segments", "qlora_debug_few_split",
    "qlora_lora_merge_workspace", "qlora_lora_merge_requantize", "qlora_adamw_step",
    "qlora_q4_table", "qlora_q4_quantize", "qlora_q4_dequantize", "qlora_q4_linear_fwd_workspace",
    "qlora_q4_linear_bwd_workspace", "qlora_q4_linear_fwd", "qlora_q4_linear_bwd",
    "qlora_group_fwd_workspace", "qlora_group_bwd_workspace", "qlora_group_fwd", "qlora_group_bwd",
]

MAX_GROUP = 4

TABLE_NF4, TABLE_INT4 = 0, 1

KERNEL_KINDS = ["quantize", "dequant", "lora_pre", "fwd_gemm", "fwd_simt", "dx_gemm", "dx_simt", "grads", "optim"]


class QloraError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Nf4WeightDesc(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("absmax_q", ctypes.c_void_p), ("absmax_scale", ctypes.c_void_p),
                ("absmax_mean", ctypes.c_void_p)]


class Q4WeightDesc(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("table", ctypes.c_int32),
                ("double_quant", ctypes.c_int32), ("codes", ctypes.c_void_p), ("absmax_q", ctypes.c_void_p),
                ("absmax_scale", ctypes.c_void_p), ("absmax_mean", ctypes.c_void_p), ("absmax", ctypes.c_void_p)]


class ProjDesc(ctypes.Structure):
    _fields_ = [("w", ctypes.POINTER(Nf4WeightDesc)), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("Y", ctypes.c_void_p), ("dY", ctypes.c_void_p), ("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_LIB_PATH} is missing "
                               "(run python -m bit_quantized_lora_double_b300._build)")
        L = ctypes.CDLL(_LIB_PATH)
        i64, sz, vp, i32, f32 = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        W = ctypes.POINTER(Nf4WeightDesc)
        for n in ("qlora_nf4_codes_bytes", "qlora_nf4_absmax_count", "qlora_nf4_scale_count",
                  "qlora_nf4_storage_bytes", "qlora_nf4_quantize_workspace"):
            getattr(L, n).restype = sz
            getattr(L, n).argtypes = [i64, i64]
        L.qlora_nf4_table.restype = None
        L.qlora_nf4_table.argtypes = [vp]
        L.qlora_nf4_quantize.restype = i32
        L.qlora_nf4_quantize.argtypes = [vp, W, vp, sz, vp]
        L.qlora_nf4_quantize_noalloc.restype = i32
        L.qlora_nf4_quantize_noalloc.argtypes = [vp, W, vp]
        L.qlora_nf4_dequantize.restype = i32
        L.qlora_nf4_dequantize.argtypes = [W, vp, vp]
        L.qlora_linear_fwd_workspace.restype = sz
        L.qlora_linear_fwd_workspace.argtypes = [i64, W, i32]
        L.qlora_linear_bwd_workspace.restype = sz
        L.qlora_linear_bwd_workspace.argtypes = [i64, W, i32]
        L.qlora_linear_fwd.restype = i32
        L.qlora_linear_fwd.argtypes = [vp, i64, W, vp, vp, i32, f32, vp, vp, vp, sz, vp]
        L.qlora_linear_bwd.restype = i32
        L.qlora_linear_bwd.argtypes = [vp, vp, vp, i64, W, vp, vp, i32, f32, vp, vp, vp, vp, sz, vp]
        L.qlora_last_error.restype = ctypes.c_char_p
        L.qlora_last_error.argtypes = []
        L.qlora_check_device_status.restype = i32
        L.qlora_check_device_status.argtypes = [vp]
        L.qlora_set_wait_limit.restype = None
        L.qlora_set_wait_limit.argtypes = [i64]
        L.qlora_version.restype = ctypes.c_char_p
        L.qlora_version.argtypes = []
        L.qlora_profile_start.restype = None
        L.qlora_profile_start.argtypes = []
        L.qlora_profile_stop.restype = i32
        L.qlora_profile_stop.argtypes = [vp, vp]
        L.qlora_lora_merge_workspace.restype = sz
        L.qlora_lora_merge_workspace.argtypes = [i64, i64]
        L.qlora_lora_merge_requantize.restype = i32
        L.qlora_lora_merge_requantize.argtypes = [W, vp, vp, i32, f32, W, vp, sz, vp]
        L.qlora_adamw_step.restype = i32
        L.qlora_adamw_step.argtypes = [vp, vp, vp, vp, vp, i64, f32, f32, f32, f32, f32, i64, vp]
        Q = ctypes.POINTER(Q4WeightDesc)
        L.qlora_q4_table.restype = None
        L.qlora_q4_table.argtypes = [i32, vp]
        L.qlora_q4_quantize.restype = i32
        L.qlora_q4_quantize.argtypes = [vp, Q, vp, sz, vp]
        L.qlora_q4_dequantize.restype = i32
        L.qlora_q4_dequantize.argtypes = [Q, vp, vp]
        L.qlora_q4_linear_fwd_workspace.restype = sz
        L.qlora_q4_linear_fwd_workspace.argtypes = [i64, Q, i32]
        L.qlora_q4_linear_bwd_workspace.restype = sz
        L.qlora_q4_linear_bwd_workspace.argtypes = [i64, Q, i32]
        L.qlora_q4_linear_fwd.restype = i32
        L.qlora_q4_linear_fwd.argtypes = [vp, i64, Q, vp, vp, i32, f32, vp, vp, vp, sz, vp]
        L.qlora_q4_linear_bwd.restype = i32
        L.qlora_q4_linear_bwd.argtypes = [vp, vp, vp, i64, Q, vp, vp, i32, f32, vp, vp, vp, vp, sz, vp]
        P = ctypes.POINTER(ProjDesc)
        for n in ("qlora_group_fwd_workspace", "qlora_group_bwd_workspace"):
            getattr(L, n).restype = sz
            getattr(L, n).argtypes = [i64, P, i32, i32]
        L.qlora_group_fwd.restype = i32
        L.qlora_group_fwd.argtypes = [vp, i64, P, i32, i32, f32, vp, vp, sz, vp]
        L.qlora_group_bwd.restype = i32
        L.qlora_group_bwd.argtypes = [vp, vp, i64, P, i32, i32, f32, vp, vp, sz, vp]
        L.qlora_debug_gemm_segments.restype = i64
        L.qlora_debug_gemm_segments.argtypes = [i64, i64, i64, i32, i32, vp, i64]
        L.qlora_debug_few_split.restype = i64
        L.qlora_debug_few_split.argtypes = [i64, i64, i64, vp, i64]
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise QloraError(status, lib().qlora_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    h = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(h)


@dataclass
class Nf4Weight:
    """A quantized weight: device arrays (torch-owned) plus the C descriptor."""
    rows: int
    cols: int
    codes: torch.Tensor
    absmax_q: torch.Tensor
    absmax_scale: torch.Tensor
    absmax_mean: torch.Tensor

    @property
    def desc(self) -> Nf4WeightDesc:
        return Nf4WeightDesc(self.rows, self.cols, self.codes.data_ptr(), self.absmax_q.data_ptr(),
                             self.absmax_scale.data_ptr(), self.absmax_mean.data_ptr())


@dataclass
class Q4Weight:
    """A quantized weight of either level table, with the block absmax
    double-quantized (absmax_q, absmax_scale, absmax_mean) or as fp32
    (absmax); the unused arrays are None."""
    rows: int
    cols: int
    table: int
    double_quant: bool
    codes: torch.Tensor
    absmax_q: Optional[torch.Tensor] = None
    absmax_scale: Optional[torch.Tensor] = None
    absmax_mean: Optional[torch.Tensor] = None
    absmax: Optional[torch.Tensor] = None

    @property
    def desc(self) -> Q4WeightDesc:
        p = lambda t: None if t is None else t.data_ptr()
        return Q4WeightDesc(self.rows, self.cols, self.table, int(self.double_quant), self.codes.data_ptr(),
                            p(self.absmax_q), p(self.absmax_scale), p(self.absmax_mean), p(self.absmax))


# ---- sizes -----------------------------------------------------------------

def qlora_nf4_codes_bytes(rows, cols):
    return lib().qlora_nf4_codes_bytes(rows, cols)


def qlora_nf4_absmax_count(rows, cols):
    return lib().qlora_nf4_absmax_count(rows, cols)


def qlora_nf4_scale_count(rows, cols):
    return lib().qlora_nf4_scale_count(rows, cols)


def qlora_nf4_storage_bytes(rows, cols):
    return lib().qlora_nf4_storage_bytes(rows, cols)


def qlora_nf4_quantize_workspace(rows, cols):
    return lib().qlora_nf4_quantize_workspace(rows, cols)


def qlora_nf4_table():
    import numpy as np
    out = np.zeros(16, np.float32)
    lib().qlora_nf4_table(out.ctypes.data_as(ctypes.c_void_p))
    return out


def qlora_q4_table(table: int):
    import numpy as np
    out = np.zeros(16, np.float32)
    lib().qlora_q4_table(int(table), out.ctypes.data_as(ctypes.c_void_p))
    return out


def qlora_q4_linear_fwd_workspace(M, w: Q4Weight, r):
    d = w.desc
    return lib().qlora_q4_linear_fwd_workspace(M, ctypes.byref(d), r)


def qlora_q4_linear_bwd_workspace(M, w: Q4Weight, r):
    d = w.desc
    return lib().qlora_q4_linear_bwd_workspace(M, ctypes.byref(d), r)


def qlora_linear_fwd_workspace(M, w: Nf4Weight, r):
    d = w.desc
    return lib().qlora_linear_fwd_workspace(M, ctypes.byref(d), r)


def qlora_linear_bwd_workspace(M, w: Nf4Weight, r):
    d = w.desc
    return lib().qlora_linear_bwd_workspace(M, ctypes.byref(d), r)


def alloc_nf4_weight(rows: int, cols: int, device="cuda") -> Nf4Weight:
    """Allocates the device arrays of a quantized weight (torch tensors)."""
    nb = qlora_nf4_absmax_count(rows, cols)
    if qlora_nf4_codes_bytes(rows, cols) == 0 and rows != 0:
        raise QloraError(2, f"invalid weight shape [{rows}, {cols}]")
    return Nf4Weight(rows, cols,
                     torch.empty(rows * cols // 2, dtype=torch.uint8, device=device),
                     torch.empty(nb, dtype=torch.int8, device=device),
                     torch.empty(qlora_nf4_scale_count(rows, cols), dtype=torch.float32, device=device),
                     torch.empty(4, dtype=torch.float32, device=device))


def alloc_q4_weight(rows: int, cols: int, table: int, double_quant: bool, device="cuda") -> Q4Weight:
    """Allocates the device arrays of a quantized weight of the given format."""
    nb = qlora_nf4_absmax_count(rows, cols)
    if qlora_nf4_codes_bytes(rows, cols) == 0 and rows != 0:
        raise QloraError(2, f"invalid weight shape [{rows}, {cols}]")
    codes = torch.empty(rows * cols // 2, dtype=torch.uint8, device=device)
    if double_quant:
        return Q4Weight(rows, cols, table, True, codes,
                        absmax_q=torch.empty(nb, dtype=torch.int8, device=device),
                        absmax_scale=torch.empty(qlora_nf4_scale_count(rows, cols), dtype=torch.float32,
                                                 device=device),
                        absmax_mean=torch.empty(4, dtype=torch.float32, device=device))
    return Q4Weight(rows, cols, table, False, codes, absmax=torch.empty(max(nb, 4), dtype=torch.float32,
                                                                         device=device))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# ---- calls -----------------------------------------------------------------

def qlora_nf4_quantize(W: torch.Tensor, out: Nf4Weight, ws: torch.Tensor, stream=None):
    d = out.desc
    _check(lib().qlora_nf4_quantize(_ptr(W), ctypes.byref(d), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)))


def qlora_nf4_quantize_noalloc(W: torch.Tensor, out: Nf4Weight, stream=None):
    """Quantize with the library's built-in scratch (no workspace, no allocation)."""
    d = out.desc
    _check(lib().qlora_nf4_quantize_noalloc(_ptr(W), ctypes.byref(d), _stream(stream)))


def qlora_nf4_dequantize(w: Nf4Weight, out: torch.Tensor, stream=None):
    d = w.desc
    _check(lib().qlora_nf4_dequantize(ctypes.byref(d), _ptr(out), _stream(stream)))


def qlora_linear_fwd(X, M, w: Nf4Weight, A, B, r, scale, Y, U_save, ws, stream=None):
    d = w.desc
    _check(lib().qlora_linear_fwd(_ptr(X), M, ctypes.byref(d), _ptr(A), _ptr(B), r, float(scale), _ptr(Y),
                                  _ptr(U_save), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream)))


def qlora_linear_bwd(dY, X, U_saved, M, w: Nf4Weight, A, B, r, scale, dX, dA, dB, ws, stream=None):
    d = w.desc
    _check(lib().qlora_linear_bwd(_ptr(dY), _ptr(X), _ptr(U_saved), M, ctypes.byref(d), _ptr(A), _ptr(B), r,
                                  float(scale), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def qlora_q4_quantize(W: torch.Tensor, out: Q4Weight, ws, stream=None):
    """Quantize into `out`'s format; `ws` may be None when out.double_quant is False."""
    d = out.desc
    _check(lib().qlora_q4_quantize(_ptr(W), ctypes.byref(d), _ptr(ws),
                                   0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def qlora_q4_dequantize(w: Q4Weight, out: torch.Tensor, stream=None):
    d = w.desc
    _check(lib().qlora_q4_dequantize(ctypes.byref(d), _ptr(out), _stream(stream)))


def qlora_q4_linear_fwd(X, M, w: Q4Weight, A, B, r, scale, Y, U_save, ws, stream=None):
    d = w.desc
    _check(lib().qlora_q4_linear_fwd(_ptr(X), M, ctypes.byref(d), _ptr(A), _ptr(B), r, float(scale), _ptr(Y),
                                     _ptr(U_save), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                     _stream(stream)))


def qlora_q4_linear_bwd(dY, X, U_saved, M, w: Q4Weight, A, B, r, scale, dX, dA, dB, ws, stream=None):
    d = w.desc
    _check(lib().qlora_q4_linear_bwd(_ptr(dY), _ptr(X), _ptr(U_saved), M, ctypes.byref(d), _ptr(A), _ptr(B), r,
                                     float(scale), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


# ---- projection groups --------------------------------------------------------

def _projs(ws_, As, Bs, Ys=None, dYs=None, dAs=None, dBs=None):
    """A ctypes array of projection descriptors (it keeps the weight
    descriptors it points to alive)."""
    n = len(ws_)
    descs = [w.desc for w in ws_]
    arr = (ProjDesc * n)()
    for g in range(n):
        arr[g].w = ctypes.pointer(descs[g])
        arr[g].A = As[g].data_ptr()
        arr[g].B = Bs[g].data_ptr()
        arr[g].Y = Ys[g].data_ptr() if Ys is not None else None
        arr[g].dY = dYs[g].data_ptr() if dYs is not None else None
        arr[g].dA = dAs[g].data_ptr() if dAs is not None else None
        arr[g].dB = dBs[g].data_ptr() if dBs is not None else None
    arr._keep = descs
    return arr


def qlora_group_fwd_workspace(M, ws_, As, Bs, r):
    return lib().qlora_group_fwd_workspace(M, _projs(ws_, As, Bs), len(ws_), r)


def qlora_group_bwd_workspace(M, ws_, As, Bs, r):
    return lib().qlora_group_bwd_workspace(M, _projs(ws_, As, Bs), len(ws_), r)


def qlora_group_fwd(X, M, ws_, As, Bs, r, scale, Ys, U_save, ws, stream=None):
    """Forward of the projections (weights ws_, adapters As, Bs) sharing X; U_save [M, n r] or None."""
    p = _projs(ws_, As, Bs, Ys=Ys)
    _check(lib().qlora_group_fwd(_ptr(X), M, p, len(ws_), r, float(scale), _ptr(U_save), _ptr(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def qlora_group_bwd(X, U_saved, M, ws_, As, Bs, r, scale, dYs, dX, dAs, dBs, ws, stream=None):
    """Backward of the projections: dA_g, dB_g and dX = the sum over g of the input gradients."""
    p = _projs(ws_, As, Bs, dYs=dYs, dAs=dAs, dBs=dBs)
    _check(lib().qlora_group_bwd(_ptr(X), _ptr(U_saved), M, p, len(ws_), r, float(scale), _ptr(dX), _ptr(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def qlora_lora_merge_workspace(rows, cols):
    return lib().qlora_lora_merge_workspace(rows, cols)


def qlora_lora_merge_requantize(w: Nf4Weight, A, B, r, scale, out: Nf4Weight, ws, stream=None):
    """Merge the adapter into the base and quantize the merged weight into `out` (may be `w`)."""
    dw, do = w.desc, out.desc
    _check(lib().qlora_lora_merge_requantize(ctypes.byref(dw), _ptr(A), _ptr(B), r, float(scale), ctypes.byref(do),
                                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def qlora_adamw_step(param, param_bf16, grad, m, v, lr, beta1, beta2, eps, weight_decay, step, stream=None):
    """One AdamW step on fp32 `param` (flat), state `m`, `v` anywhere the device can reach."""
    _check(lib().qlora_adamw_step(_ptr(param), _ptr(param_bf16), _ptr(grad), _ptr(m), _ptr(v), param.numel(),
                                  float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step),
                                  _stream(stream)))


def qlora_last_error() -> str:
    return lib().qlora_last_error().decode()


def qlora_check_device_status(stream=None):
    _check(lib().qlora_check_device_status(_stream(stream)))


def qlora_set_wait_limit(microseconds: int):
    lib().qlora_set_wait_limit(int(microseconds))


def qlora_version() -> str:
    return lib().qlora_version().decode()


def qlora_debug_gemm_segments(M: int, Nd: int, nk_main: int, lora_steps: int, pairs_resident: int):
    """The fused GEMM's work schedule (host computation, no GPU): returns
    (tile_rows, dp_tiles, pairs, tiles, records), records an int64 array of
    rows (pair, tile, row0, col0, kbeg, nk, role, head, contributors); see the
    C header for the fields. Raises QloraError(QLORA_ERR_SHAPE) on bad input."""
    import numpy as np
    cap = 4 + 9 * 4096
    while True:
        out = np.zeros(cap, np.int64)
        n = lib().qlora_debug_gemm_segments(int(M), int(Nd), int(nk_main), int(lora_steps), int(pairs_resident),
                                            out.ctypes.data, cap)
        if n >= 0:
            return int(out[0]), int(out[1]), int(out[2]), int(out[3]), out[4:4 + 9 * n].reshape(n, 9).copy()
        if n != -1:
            raise QloraError(2, "qlora_debug_gemm_segments: invalid arguments")
        cap *= 4


def qlora_debug_few_split(M: int, N: int, K: int):
    """The few-token forward's split of an N x K weight for M tokens (host
    computation, no GPU): returns (tasks, warps, P, tiles, ranges, tile_warps), ranges an
    int64 array [warps, 2] of each warp's task range [first, end) and
    tile_warps [tiles, 2] each row tile's first and last contributing warp.
    Raises QloraError(QLORA_ERR_SHAPE) on bad input."""
    import numpy as np
    cap = 4 + 2 * 16 * 148 + 2 * ((int(N) + 31) // 32)
    out = np.zeros(cap, np.int64)
    n = lib().qlora_debug_few_split(int(M), int(N), int(K), out.ctypes.data, cap)
    if n < 0:
        raise QloraError(2, "qlora_debug_few_split: invalid arguments")
    T, W, P, tiles = (int(v) for v in out[:4])
    return (T, W, P, tiles, out[4:4 + 2 * W].reshape(W, 2).copy(),
            out[4 + 2 * W:4 + 2 * W + 2 * tiles].reshape(tiles, 2).copy())


def qlora_profile_start():
    lib().qlora_profile_start()


def qlora_profile_stop():
    """Returns ({kind: summed ms}, {kind: launches}, total launches)."""
    import numpy as np
    ms = np.zeros(len(KERNEL_KINDS), np.float64)
    n = np.zeros(len(KERNEL_KINDS), np.int32)
    total = lib().qlora_profile_stop(ms.ctypes.data_as(ctypes.c_void_p), n.ctypes.data_as(ctypes.c_void_p))
    if total < 0:
        raise QloraError(6, "profiling events failed")
    return dict(zip(KERNEL_KINDS, ms.tolist())), dict(zip(KERNEL_KINDS, n.tolist())), int(total)
