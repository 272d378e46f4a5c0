"""The fused GEMM's work schedule, checked on the host (no GPU).

The tensor-core GEMM runs on a persistent grid of CTA pairs: whole output
tiles data-parallel, then a stream-K line in which a pair starting inside a
tile computes its tail (an fp32 partial) and the pair holding the tile's first
k-steps finishes it with the following pairs' tails. The kernel's four roles
(TMA producer, MMA issuer, decoders, epilogue) walk the same segments; the
library exports a host enumeration built from those very functions. A wrong
schedule would drop or double a k-step (wrong output) or make a finishing
pair wait for a tail nobody writes (a bounded wait that runs out), so the
invariants are checked here over many shapes and pair counts.
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
    for q, t, m0, c0, kb, nk, role, ce in rec.tolist():
        assert 0 <= q < P and 0 <= t < T and nk >= 1 and 0 <= kb and kb + nk <= S
        assert m0 % tile_rows == 0 and 0 <= m0 < M and c0 % BN == 0 and 0 <= c0 < Nd
        # one (row, column) origin per tile, and no two tiles share one
        assert origin.setdefault(t, (m0, c0)) == (m0, c0)
        cover[t, kb:kb + nk] += 1
        by_pair.setdefault(q, []).append((t, kb, nk, role, ce))
        full = kb == 0 and nk == S
        assert role == (0 if full else (1 if kb == 0 else 2))
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
    # each head's contributors hold exactly the rest of its tile, as tails
    n_heads = 0
    for q, (t, kb, nk, role, ce) in last.items():
        if role != 1:
            continue
        n_heads += 1
        assert q + 1 < ce <= P
        pieces = [(kb, nk)]
        for c in range(q + 1, ce):
            tc, kbc, nkc, rolec, _ = first_sk[c]
            assert tc == t and rolec == 2
            pieces.append((kbc, nkc))
        pieces.sort()
        assert pieces[0][0] == 0 and sum(p[1] for p in pieces) == S
        assert all(a[0] + a[1] == b[0] for a, b in zip(pieces, pieces[1:]))
    # every tail is consumed by some head
    for c, s in first_sk.items():
        if s is not None and s[3] == 2:
            assert any(last[q][3] == 1 and last[q][0] == s[0] and q < c < last[q][4] for q in last)
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
    assert check(32768, 14336, 64, 1, 74)[:4] == (512, 3478, 74, 3584)


def test_rejects_bad_arguments():
    with pytest.raises(qlora.QloraError):
        qlora.qlora_debug_gemm_segments(0, 256, 64, 1, 74)
    with pytest.raises(qlora.QloraError):
        qlora.qlora_debug_gemm_segments(256, 256, 64, 1, 75)
