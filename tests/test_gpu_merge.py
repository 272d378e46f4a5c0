"""GPU parity of the adapter merge + requantization: the merged NF4 weight
(codes, int8 absmax codes, scales, mean) and its dequantized values must equal
the oracle's bit for bit (xingyuzhitong.com "Fine-Tuning Memory
Requirements", section "Choosing a method")."""
import numpy as np
import pytest
import torch

from bit_quantized_lora_double_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


@pytest.mark.parametrize("N,K,r,scale,inplace", [
    (64, 128, 8, 2.0, False),
    (257, 1024, 5, 0.5, False),      # rank not a multiple of 8, partial DQ group
    (1000, 192, 64, 0.25, True),     # in place (out is the base weight)
    (512, 4096, 128, 1.0, False),    # largest rank
])
def test_merge_requantize_bit_exact(g, oracle, N, K, r, scale, inplace):
    from bit_quantized_lora_double_b300 import qlora
    from tests.test_gpu_codec import assert_quant_equal
    W = synth.gaussian_bf16((N, K), 0.02, 8000 + N)
    A = synth.gaussian_bf16((r, K), 1.0 / 32, 8001 + N)
    B = synth.gaussian_bf16((N, r), 0.05, 8002 + N)
    qw = oracle.nf4_quantize(W)
    w = g.weight_from_oracle(qw)
    out = w if inplace else qlora.alloc_nf4_weight(N, K)
    ws = qlora.workspace(qlora.qlora_lora_merge_workspace(N, K))
    qlora.qlora_lora_merge_requantize(w, g.dev_bf16(A), g.dev_bf16(B), r, scale, out, ws)
    torch.cuda.synchronize()
    merged = oracle.lora_merge(oracle.nf4_dequantize(qw), A, B, scale)
    assert np.array_equal(g.host_u16(ws[:N * K * 2].view(torch.int16).view(N, K).view(torch.bfloat16)), merged)
    ref = oracle.nf4_quantize(merged)
    assert_quant_equal(out, ref)
    assert np.array_equal(g.dequantize(out), oracle.nf4_dequantize(ref))
