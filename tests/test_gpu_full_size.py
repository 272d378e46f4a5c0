"""GPU parity at the full workload shapes the benchmark times, on sampled rows.

The layer calls run on the whole problem (every token, every output column),
in the same launch configuration as the benchmark (forward with U saved, then
the backward with that U). The oracle then computes, one by one, a fixed set of
256 token rows of Y and dX, and dA, dB and U in full (they are sums over all
tokens). Bars as in the other parity tests: NF4 codes bit-exact against the
oracle's quantizer; relative Frobenius error <= 5e-3 per output tensor.

Shapes (N out x K in, M tokens, rank r, scale s = alpha / r):
  Llama-3.1-8B gate 14336 x 4096 and down 4096 x 14336, M = 2048, r = 16, s = 2;
  Llama-70B gate 28672 x 8192 and down 8192 x 28672, M = 4096, r = 64, s = 0.25;
  gate 14336 x 4096 at M = 32768, r = 16, s = 2;
  the forward alone at M = 1 and 16 tokens with K = 28672 (70B down).
Inputs follow the seeded recipe of synth.layer_inputs for each workload.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 5e-3
SAMPLE_ROWS = 256


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


def sample_rows(M, seed):
    """256 sorted token rows (all of them when M <= 256), always with the first and last."""
    if M <= SAMPLE_ROWS:
        return np.arange(M)
    rows = np.random.default_rng(seed).choice(np.arange(1, M - 1), SAMPLE_ROWS - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], rows]))


def quantize_checked(g, oracle, W):
    w = g.quantize(W)
    qw = oracle.nf4_quantize(W)
    assert np.array_equal(w.codes.cpu().numpy(), qw["codes"]), "NF4 codes differ"
    assert np.array_equal(w.absmax_q.cpu().numpy(), qw["absmax_q"]), "int8 absmax codes differ"
    return w, oracle.nf4_dequantize(qw)


CASES = [
    # id, workload, projection index, M
    ("llama8b-gate-M2048", 1, 4, None),
    ("llama8b-down-M2048", 1, 6, None),
    ("llama70b-gate-M4096", 3, 4, None),
    ("llama70b-down-M4096", 3, 6, None),
    ("gate-sweep-M32768", 4, 0, 32768),
]


@pytest.mark.parametrize("name,wl,proj,M", CASES, ids=[c[0] for c in CASES])
def test_full_size_fwd_bwd(g, oracle, name, wl, proj, M):
    X, W, A, B, dY, s = synth.layer_inputs(wl, proj, M=M)
    M, r = X.shape[0], A.shape[0]
    w, Wdq = quantize_checked(g, oracle, W)
    del W
    Y, U = g.fwd(X, w, A, B, r, s)
    dX, dA, dB = g.bwd(dY, X, U, w, A, B, r, s)
    rows = sample_rows(M, 100 * wl + proj)
    Yr, Ur = oracle.linear_fwd(X, Wdq, A, B, s, rows=rows)
    dXr, dAr, dBr = oracle.linear_bwd(dY, X, Wdq, A, B, s, rows=rows)
    import torch
    ri = torch.from_numpy(rows).cuda()
    errs = {
        "Y": g.rel_fro(g.host_f64_bf16(Y.index_select(0, ri)), Yr),
        "U": g.rel_fro(g.host_f64_bf16(U), Ur),
        "dX": g.rel_fro(g.host_f64_bf16(dX.index_select(0, ri)), dXr),
        "dA": g.rel_fro(dA.cpu().numpy(), dAr),
        "dB": g.rel_fro(dB.cpu().numpy(), dBr),
    }
    for k, v in errs.items():
        assert v <= TOL, (name, k, v, errs)


@pytest.mark.parametrize("M", [1, 16])
def test_full_size_forward_few_tokens_long_k(g, oracle, M):
    # 70B down projection (K = 28672, beyond the few-token kernel's table of
    # reconstructed absmax values) with one and sixteen tokens
    X, W, A, B, _, s = synth.layer_inputs(3, 6, M=M)
    r = A.shape[0]
    w, Wdq = quantize_checked(g, oracle, W)
    Y, U = g.fwd(X, w, A, B, r, s)
    Yr, Ur = oracle.linear_fwd(X, Wdq, A, B, s)
    assert g.rel_fro(g.host_f64_bf16(Y), Yr) <= TOL
    assert g.rel_fro(g.host_f64_bf16(U), Ur) <= TOL
