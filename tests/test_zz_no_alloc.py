"""The quantizer variant that allocates nothing: qlora_nf4_quantize_noalloc.

It serves callers that cannot allocate device memory (a plugin whose host
application owns every device buffer, or code that must not trigger
cudaMalloc's implicit synchronization mid-run). It takes no workspace and uses
the library's built-in scratch array instead. Called through the C ABI, it
must give the same bytes as qlora_nf4_quantize with a caller workspace, on two
calls in a row (the second call finds the first call's data in the shared
scratch and must not depend on it). This file sorts last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _arrays(w):
    return (w.codes.cpu().numpy(), w.absmax_q.cpu().numpy(), w.absmax_scale.cpu().numpy().view(np.uint32),
            np.float32(w.absmax_mean[0].item()).view(np.uint32))


def test_noalloc_matches_workspace_quantize_two_calls():
    import torch
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from bit_quantized_lora_double_b300 import qlora, synth

    L = qlora.lib()
    for call, (rows, cols) in enumerate([(257, 1024), (4096, 4096 + 3 * 64)]):
        W = synth.gaussian_bf16((rows, cols), 0.02, 9100 + call)
        Wd = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).cuda()
        ref = qlora.alloc_nf4_weight(rows, cols)
        qlora.qlora_nf4_quantize(Wd, ref, qlora.workspace(qlora.qlora_nf4_quantize_workspace(rows, cols)))
        got = qlora.alloc_nf4_weight(rows, cols)
        d = got.desc
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        status = L.qlora_nf4_quantize_noalloc(ctypes.c_void_p(Wd.data_ptr()), ctypes.byref(d), stream)
        assert status == 0, qlora.qlora_last_error()
        torch.cuda.synchronize()
        qlora.qlora_check_device_status()
        for a, b in zip(_arrays(got), _arrays(ref)):
            assert np.array_equal(a, b)


def test_noalloc_rejects_weight_beyond_scratch():
    from bit_quantized_lora_double_b300 import qlora
    L = qlora.lib()
    rows, cols = 65536, 8192  # needs about 32 MiB of scratch
    assert qlora.qlora_nf4_quantize_workspace(rows, cols) > 16 * 1024 * 1024
    fake = 1 << 20
    d = qlora.Nf4WeightDesc(rows, cols, fake, fake, fake, fake)
    assert L.qlora_nf4_quantize_noalloc(ctypes.c_void_p(fake), ctypes.byref(d), None) == 4
    assert "scratch" in qlora.qlora_last_error()
