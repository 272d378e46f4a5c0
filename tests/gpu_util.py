"""Helpers for the GPU parity tests: moving bf16 bit arrays to and from the
device, calling the library through its binding, and the error measure."""
import numpy as np
import torch

from bit_quantized_lora_double_b300 import qlora, synth


def dev_bf16(h: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(h, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64_bf16(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits_to_f32(host_u16(t)).astype(np.float64)


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(np.asarray(got, np.float64) - ref) / (den if den > 0 else 1.0))


def quantize(W: np.ndarray):
    rows, cols = W.shape
    w = qlora.alloc_nf4_weight(rows, cols)
    ws = qlora.workspace(qlora.qlora_nf4_quantize_workspace(rows, cols))
    qlora.qlora_nf4_quantize(dev_bf16(W), w, ws)
    return w


def weight_from_oracle(qw: dict):
    """Device copy of an oracle-quantized weight (to test decode alone)."""
    w = qlora.alloc_nf4_weight(qw["rows"], qw["cols"])
    w.codes.copy_(torch.from_numpy(qw["codes"]))
    w.absmax_q.copy_(torch.from_numpy(qw["absmax_q"]))
    w.absmax_scale.copy_(torch.from_numpy(qw["absmax_scale"]))
    w.absmax_mean[0] = float(qw["absmax_mean"])
    return w


TABLES = {"nf4": qlora.TABLE_NF4, "int4": qlora.TABLE_INT4}


def q4_quantize(W: np.ndarray, table: str, double_quant: bool):
    rows, cols = W.shape
    w = qlora.alloc_q4_weight(rows, cols, TABLES[table], double_quant)
    ws = qlora.workspace(qlora.qlora_nf4_quantize_workspace(rows, cols)) if double_quant else None
    qlora.qlora_q4_quantize(dev_bf16(W), w, ws)
    return w


def q4_weight_from_oracle(qw: dict):
    """Device copy of an oracle-quantized weight of any format."""
    w = qlora.alloc_q4_weight(qw["rows"], qw["cols"], TABLES[qw["table"]], qw["double_quant"])
    w.codes.copy_(torch.from_numpy(qw["codes"]))
    if qw["double_quant"]:
        w.absmax_q.copy_(torch.from_numpy(qw["absmax_q"]))
        w.absmax_scale.copy_(torch.from_numpy(qw["absmax_scale"]))
        w.absmax_mean[0] = float(qw["absmax_mean"])
    else:
        w.absmax[:len(qw["absmax"])].copy_(torch.from_numpy(qw["absmax"]))
    return w


def _is_q4(w) -> bool:
    return isinstance(w, qlora.Q4Weight)


def dequantize(w) -> np.ndarray:
    out = torch.empty((w.rows, w.cols), dtype=torch.bfloat16, device="cuda")
    (qlora.qlora_q4_dequantize if _is_q4(w) else qlora.qlora_nf4_dequantize)(w, out)
    torch.cuda.synchronize()
    return host_u16(out)


def fwd(X, w, A, B, r, scale, save_u=True):
    M = X.shape[0]
    Xd, Ad, Bd = dev_bf16(X), dev_bf16(A), dev_bf16(B)
    Y = torch.empty((M, w.rows), dtype=torch.bfloat16, device="cuda")
    U = torch.empty((M, r), dtype=torch.bfloat16, device="cuda") if save_u else None
    if _is_q4(w):
        ws = qlora.workspace(qlora.qlora_q4_linear_fwd_workspace(M, w, r))
        qlora.qlora_q4_linear_fwd(Xd, M, w, Ad, Bd, r, scale, Y, U, ws)
    else:
        ws = qlora.workspace(qlora.qlora_linear_fwd_workspace(M, w, r))
        qlora.qlora_linear_fwd(Xd, M, w, Ad, Bd, r, scale, Y, U, ws)
    torch.cuda.synchronize()
    qlora.qlora_check_device_status()
    return Y, U


def bwd(dY, X, U, w, A, B, r, scale):
    M = X.shape[0]
    dX = torch.empty((M, w.cols), dtype=torch.bfloat16, device="cuda")
    dA = torch.empty((r, w.cols), dtype=torch.float32, device="cuda")
    dB = torch.empty((w.rows, r), dtype=torch.float32, device="cuda")
    if _is_q4(w):
        ws = qlora.workspace(qlora.qlora_q4_linear_bwd_workspace(M, w, r))
        qlora.qlora_q4_linear_bwd(dev_bf16(dY), dev_bf16(X), U, M, w, dev_bf16(A), dev_bf16(B), r, scale, dX, dA,
                                  dB, ws)
    else:
        ws = qlora.workspace(qlora.qlora_linear_bwd_workspace(M, w, r))
        qlora.qlora_linear_bwd(dev_bf16(dY), dev_bf16(X), U, M, w, dev_bf16(A), dev_bf16(B), r, scale, dX, dA, dB,
                               ws)
    torch.cuda.synchronize()
    qlora.qlora_check_device_status()
    return dX, dA, dB
