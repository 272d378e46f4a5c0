"""Two layer calls on two CUDA streams at once, both on the fused tensor-core
GEMM with stream-K tiles (work shared between CTA pairs).

Each launch is sized for the whole GPU, so while both are queued the GPU runs
some pairs of one and some of the other, and a pair of either may start only
after pairs of the other have finished. A shared tile is finished by whichever
of its contributors arrives last, never by a pair waiting for one that has not
started, so both calls must complete with correct results and no bounded wait
may run out. Outputs are checked against the oracle on sampled rows (Y, dX)
and in full (dA, dB), relative Frobenius error <= 5e-3, after the calls have
run several times interleaved. The partials of a shared tile are added in
pair order whichever contributor finishes it, so the outputs must also equal,
bit for bit, those of the same calls run alone.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import qlora, synth

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def g():
    from bit_quantized_lora_double_b300 import _build
    _build.build()
    from tests import gpu_util
    return gpu_util


class Problem:
    def __init__(self, g, oracle, M, N, K, r, scale, seed):
        import torch
        self.M, self.N, self.K, self.r, self.scale = M, N, K, r, scale
        self.X = synth.gaussian_bf16((M, K), 1.0, seed)
        W = synth.gaussian_bf16((N, K), 0.02, seed + 1)
        self.A = synth.gaussian_bf16((r, K), 1.0 / K, seed + 2)
        self.B = synth.gaussian_bf16((N, r), 0.01, seed + 3)
        self.dY = synth.gaussian_bf16((M, N), 1.0, seed + 4)
        qw = oracle.nf4_quantize(W)
        self.Wdq = oracle.nf4_dequantize(qw)
        self.w = g.weight_from_oracle(qw)
        d = g.dev_bf16
        self.Xd, self.Ad, self.Bd, self.dYd = d(self.X), d(self.A), d(self.B), d(self.dY)
        self.Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        self.U = torch.empty((M, r), dtype=torch.bfloat16, device="cuda")
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
        self.dA = torch.empty((r, K), dtype=torch.float32, device="cuda")
        self.dB = torch.empty((N, r), dtype=torch.float32, device="cuda")
        self.wsf = qlora.workspace(qlora.qlora_linear_fwd_workspace(M, self.w, r))
        self.wsb = qlora.workspace(qlora.qlora_linear_bwd_workspace(M, self.w, r))

    def run(self, stream):
        qlora.qlora_linear_fwd(self.Xd, self.M, self.w, self.Ad, self.Bd, self.r, self.scale, self.Y, self.U,
                               self.wsf, stream)
        qlora.qlora_linear_bwd(self.dYd, self.Xd, self.U, self.M, self.w, self.Ad, self.Bd, self.r, self.scale,
                               self.dX, self.dA, self.dB, self.wsb, stream)

    def outputs(self):
        return [t.clone() for t in (self.Y, self.U, self.dX, self.dA, self.dB)]

    def check(self, g, oracle):
        import torch
        rows = np.sort(np.random.default_rng(self.M).choice(self.M, 128, replace=False))
        Yr, _ = oracle.linear_fwd(self.X, self.Wdq, self.A, self.B, self.scale, rows=rows)
        dXr, dAr, dBr = oracle.linear_bwd(self.dY, self.X, self.Wdq, self.A, self.B, self.scale, rows=rows)
        ri = torch.from_numpy(rows).cuda()
        errs = {
            "Y": g.rel_fro(g.host_f64_bf16(self.Y.index_select(0, ri)), Yr),
            "dX": g.rel_fro(g.host_f64_bf16(self.dX.index_select(0, ri)), dXr),
            "dA": g.rel_fro(self.dA.cpu().numpy(), dAr),
            "dB": g.rel_fro(self.dB.cpu().numpy(), dBr),
        }
        for k, v in errs.items():
            assert v <= TOL, (k, v, errs)


def test_two_streams_stream_k(g, oracle):
    import torch
    # both schedules share tiles between pairs (checked on the host below):
    # a k/v-shaped forward (8 x 4 tiles of 256 rows, stream-K over all of
    # them) and a wider one (3 x 28 tiles of 512 rows on 74 pairs, stream-K
    # over all of them too)
    a = Problem(g, oracle, 2048, 1024, 4096, 16, 2.0, 11)
    b = Problem(g, oracle, 1536, 7168, 1024, 8, 1.0, 21)
    for P in (a, b):
        _, _, _, _, rec = qlora.qlora_debug_gemm_segments(P.M, P.N, P.K // 64, 1, 74)
        assert (rec[:, 8] > 1).any(), "the forward shares tiles between pairs"
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    # alone first
    a.run(s1)
    torch.cuda.synchronize()
    b.run(s2)
    torch.cuda.synchronize()
    qlora.qlora_check_device_status()
    alone = [a.outputs(), b.outputs()]
    for _ in range(6):
        a.run(s1)
        b.run(s2)
    torch.cuda.synchronize()
    qlora.qlora_check_device_status()
    for P, ref in zip((a, b), alone):
        for name, got, want in zip(("Y", "U", "dX", "dA", "dB"), P.outputs(), ref):
            assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got.view(torch.int32),
                               want.view(torch.int16) if want.dtype == torch.bfloat16 else want.view(torch.int32)), name
    a.check(g, oracle)
    b.check(g, oracle)
