"""Host checks of the few-token forward's split of the weight (no GPU).

The kernel cuts an N x K weight into tasks of 32 rows x 256 k, numbered row
tile by row tile, and splits the line of tasks evenly over its warps; a row
tile touched by several warps is finished by the last of them to arrive, which
reads every contributor's slot: slot 1 of the first contributor when that
warp's range starts before the tile (the tile is its last), slot 0 otherwise.
These tests take the split the library computes (qlora_debug_few_split) and
check it against the definitions by brute force: every task in exactly one
range, no empty range, each tile's contributors exactly the warps whose ranges
meet it, at most two shared tiles per warp on distinct slots, and the slot the
finisher reads for each contributor equal to the slot that contributor writes.
"""
import numpy as np
import pytest

from bit_quantized_lora_double_b300 import qlora

SHAPES = [
    (14336, 4096), (4096, 14336), (4096, 4096), (1024, 4096), (6144, 4096),
    (28672, 8192), (8192, 28672), (8192, 8192), (1024, 8192),
    (1, 256), (33, 1024), (96, 4096), (700, 256), (520, 3072), (1000, 2048), (320, 256),
]
_rng = np.random.default_rng(11)
SHAPES += [(int(_rng.integers(1, 40000)), 256 * int(_rng.integers(1, 120))) for _ in range(40)]


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("N,K", SHAPES)
def test_few_split(M, N, K):
    T, W, P, tiles, rng, tw = qlora.qlora_debug_few_split(M, N, K)
    assert P == K // 256 and tiles == (N + 31) // 32 and T == tiles * P
    assert W == min(T, (16 if M <= 8 else 12) * 148)
    # even split: warp w starts at floor(w T / W); ranges tile [0, T), none empty
    w = np.arange(W, dtype=np.int64)
    assert np.array_equal(rng[:, 0], w * T // W)
    assert np.array_equal(rng[:, 1], (w + 1) * T // W)
    assert rng[0, 0] == 0 and rng[-1, 1] == T
    assert np.all(rng[:, 1] > rng[:, 0])
    assert np.array_equal(rng[1:, 0], rng[:-1, 1])
    # a tile's contributors are exactly the warps whose ranges meet it
    a = np.arange(tiles, dtype=np.int64) * P
    b = a + P
    first = np.searchsorted(rng[:, 1], a, side="right")     # first warp with end > a
    last = np.searchsorted(rng[:, 0], b, side="left") - 1   # last warp with start < b
    assert np.array_equal(tw[:, 0], first)
    assert np.array_equal(tw[:, 1], last)
    # a tile is finished by its own warp exactly when it lies inside one range
    owned = (rng[tw[:, 0], 0] <= a) & (rng[tw[:, 0], 1] >= b)
    assert np.array_equal(owned, tw[:, 0] == tw[:, 1])
    # slots: what each contributor writes equals what the finisher reads
    writes = {}
    for t in np.nonzero(~owned)[0]:
        for c in range(int(tw[t, 0]), int(tw[t, 1]) + 1):
            e = 0 if rng[c, 0] // P == t else 1           # the warp's own rule
            assert (c, e) not in writes, (N, K, c, e)      # two shared tiles of a warp never share a slot
            writes[(c, e)] = t
            read = (1 if rng[c, 0] < a[t] else 0) if c == tw[t, 0] else 0   # the finisher's rule
            assert read == e, (N, K, t, c)
    # and no warp touches more than two shared tiles
    per = np.bincount(np.array([c for c, _ in writes], dtype=np.int64), minlength=W) if writes else np.zeros(W)
    assert per.max(initial=0) <= 2


def test_few_split_rejects():
    for M, N, K in [(1, 0, 256), (1, 10, 100), (1, 10, 0), (1, 1 << 20, 1 << 20), (0, 10, 256), (17, 10, 256)]:
        with pytest.raises(qlora.QloraError):
            qlora.qlora_debug_few_split(M, N, K)
