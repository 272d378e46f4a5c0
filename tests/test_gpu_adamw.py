"""GPU AdamW step for the adapters against the fp64 oracle, with the optimizer
state in device memory and in pinned host memory ("paged optimizers":
inquiringlines.com note, mechanism paragraph; ashishsrivastav.com, section
"Paged Optimizers: Managing Fragmentation").

Bar: the GPU runs in fp32, the oracle in fp64; after three steps every
parameter and moment is within 2e-6 relative (plus 1e-9 absolute) of the
oracle's. The bf16 copy is exactly bf16_rne of the GPU's fp32 parameter.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_quantized_lora_double_b300 import synth

pytestmark = pytest.mark.gpu
HP = dict(lr=2e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module")
def q():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from bit_quantized_lora_double_b300 import qlora
    return qlora


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_adamw_matches_oracle(q, oracle, where):
    n = 10007  # a tail of n % 4 == 3
    rng = np.random.default_rng(31)
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(n) * 1e-3 * (t + 1)).astype(np.float32) for t in range(3)]
    if where == "device":
        p, m, v = (torch.from_numpy(x.copy()).cuda() for x in (p0, np.zeros(n, np.float32), np.zeros(n, np.float32)))
    else:
        p, m, v = (torch.from_numpy(x.copy()).pin_memory() for x in (p0, np.zeros(n, np.float32), np.zeros(n, np.float32)))
    pb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    rp, rm, rv = p0.astype(np.float64), np.zeros(n), np.zeros(n)
    for t, gr in enumerate(grads, 1):
        g = torch.from_numpy(gr).cuda()
        q.qlora_adamw_step(p, pb, g, m, v, step=t, **HP)
        torch.cuda.synchronize()
        oracle.adamw_step(rp, gr.astype(np.float64), rm, rv, step=t, **HP)
    for got, ref in ((p, rp), (m, rm), (v, rv)):
        got = got.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= 2e-6 * np.abs(ref) + 1e-9), np.max(np.abs(got - ref))
    pf = p.cpu().numpy()
    assert np.array_equal(pb.view(torch.int16).cpu().numpy().view(np.uint16), synth.f32_to_bf16_bits(pf))


def test_adamw_rejects_pageable_host_memory(q):
    n = 64
    p = torch.zeros(n)  # pageable host memory: the device cannot reach it
    g = torch.zeros(n, device="cuda")
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    L = q.lib()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.qlora_adamw_step(ptr(p), None, ptr(g), ptr(m), ptr(v), n, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None)
    assert st == 8 and "reachable" in q.qlora_last_error()
    assert torch.all(p == 0)
