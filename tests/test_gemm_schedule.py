"""The fused GEMM's work schedule, checked on the host (no GPU).

The tensor-core GEMM runs on a persistent grid of CTA pairs: whole output
tiles data-parallel, then a stream-K line in which the pairs sharing a tile
(its head, holding the first k-steps, and the pairs whose ranges start inside
it) each compute an fp32 partial, and whichever arrives last adds the others'
in pair order and writes the output. The kernel's four roles (TMA producer,
MMA issuer, decoders, epilogue) walk the same segments; the library exports a
host enumeration built from those very functions, with each segment's head
pair and contributor count as the epilogue computes them. A wrong schedule
would drop or double a k-step (wrong output), name a contributor that writes
no partial (a bounded wait that runs out), or share a tile among more pairs
than the epilogue's finishing ring holds, so the invariants are checked here
over many shapes and pair counts.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import qlora

BN = 256


def cdiv(a, b):
    return -(-a // b)


def check(M, Nd, nk_main, lora_steps, P_res):
    tile_rows, dpt, P, T, rec = qlora.qlora_debug_gemm_segments(M, Nd, nk_main, lora_steps, P_res)
    S = nk_main + lora_steps
    assert tile_rows in (256, 512)
    mt, nt = cdiv(M, tile_rows), cdiv(Nd, BN)
    assert T == mt * nt and 1 <= P <= P_res and 0 <= dpt <= T
    cover = np.zeros((T, S), np.int32)
    origin = {}
    first_sk, last = {}, {}
    by_pair = {}
    contrib = {}
    for q, t, m0, c0, kb, nk, role, h, n in rec.tolist():
        assert 0 <= q < P and 0 <= t < T and nk >= 1 and 0 <= kb and kb + nk <= S
        assert m0 % tile_rows == 0 and 0 <= m0 < M and c0 % BN == 0 and 0 <= c0 < Nd
        # one (row, column) origin per tile, and no two tiles share one
        assert origin.setdefault(t, (m0, c0)) == (m0, c0)
        cover[t, kb:kb + nk] += 1
        by_pair.setdefault(q, []).append((t, kb, nk, role, h, n))
        full = kb == 0 and nk == S
        assert role == (0 if full else (1 if kb == 0 else 2))
        assert (h, n) == (q, 1) if full else (h <= q < h + n and n >= 2)
        assert (role == 1) == (not full and h == q)
        contrib.setdefault(t, []).append((q, kb, nk, h, n))
    assert len(set(origin.values())) == T
    assert (cover == 1).all(), "every k-step of every tile exactly once"
    for q, segs in by_pair.items():
        dp = [s for s in segs if s[0] < dpt]
        sk = [s for s in segs if s[0] >= dpt]
        assert segs[:len(dp)] == dp, "data-parallel tiles first"
        assert [s[0] for s in dp] == list(range(q, dpt, P))
        assert all(s[3] == 0 for s in dp)
        for i, s in enumerate(sk):
            if s[3] == 2:
                assert i == 0, "a tail is the pair's first stream-K segment"
            if s[3] == 1:
                assert i == len(sk) - 1, "a head is the pair's last segment"
        first_sk[q] = sk[0] if sk else None
        last[q] = segs[-1]
    # a shared tile's contributors are pairs h .. h + n - 1, in k order, each
    # agreeing on (h, n); at most four share a tile (the epilogue's finishing
    # ring holds the pieces of up to six others)
    n_heads = 0
    for t, segs in contrib.items():
        if len(segs) == 1 and segs[0][2] == S:
            continue
        n_heads += 1
        segs.sort()
        h, n = segs[0][3], segs[0][4]
        assert all((s[3], s[4]) == (h, n) for s in segs)
        assert [s[0] for s in segs] == list(range(h, h + n)), "contributors are consecutive pairs"
        assert segs[0][1] == 0 and all(a[1] + a[2] == b[1] for a, b in zip(segs, segs[1:]))
        assert 2 <= n <= 4
    return tile_rows, dpt, P, T, n_heads


@pytest.mark.parametrize("P_res", [74, 73, 37, 5, 2, 1])
@pytest.mark.parametrize("M", [1, 64, 256, 257, 511, 512, 513, 2048, 2148, 4708, 8192])
@pytest.mark.parametrize("Nd", [8, 100, 256, 1024, 4000, 14336])
@pytest.mark.parametrize("nk", [(1, 1), (2, 1), (16, 1), (64, 1), (64, 2), (224, 1), (0, 1)])
def test_schedule_invariants(P_res, M, Nd, nk):
    check(M, Nd, nk[0], nk[1], P_res)


def test_llama8b_layer_schedules():
    """The 8B layer's GEMMs on a B300 (74 resident pairs): gate/up forward and
    down dX split into one data-parallel round and a stream-K remainder, the
    single-round shapes stay data-parallel, the small k/v forward is stream-K
    over 256-row tiles."""
    assert check(2048, 14336, 64, 1, 74)[:4] == (512, 148, 74, 224)   # gate/up fwd, down dX
    assert check(2048, 4096, 64, 1, 74)[:4] == (512, 64, 64, 64)      # q/o fwd and dX
    assert check(2048, 4096, 224, 1, 74)[:4] == (512, 64, 64, 64)     # gate/up dX, down fwd
    assert check(2048, 1024, 64, 1, 74)[:4] == (256, 0, 74, 32)       # k/v fwd
    # 48 whole rounds, then stream-K over the 32 tiles left (a share of 28
    # steps per pair, over a third of a 65-step tile)
    assert check(32768, 14336, 64, 1, 74)[:4] == (512, 3552, 74, 3584)
    # the 70B layer (M = 4096): with a 224 MiB activation (down forward, gate
    # and up dX) 3 rounds of the 256 tiles, then stream-K over 34; with a
    # 64 MiB one (q/o), which stays in L2, 2 rounds and stream-K over 108
    assert check(4096, 8192, 448, 1, 74)[:4] == (512, 222, 74, 256)
    assert check(4096, 8192, 128, 1, 74)[:4] == (512, 148, 74, 256)


def test_rejects_bad_arguments():
    with pytest.raises(qlora.QloraError):
        qlora.qlora_debug_gemm_segments(0, 256, 64, 1, 74)
    with pytest.raises(qlora.QloraError):
        qlora.qlora_debug_gemm_segments(256, 256, 64, 1, 75)
