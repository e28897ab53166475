"""The prefill kernel's split schedule, checked on the host through the
library's own index arithmetic (bitdelta_debug_split_schedule runs the same
inline functions the kernel calls; no device is used).

For a split region of sk_tiles tiles over n_pairs CTA pairs (sk_tiles >=
n_pairs): every k-block of every tile of the region is taken by exactly one
pair; a tile is either wholly one pair's or shared by exactly two, named in
k order with the slots their partials go to; no two partials share a slot;
the counter index is the tile's own and within the region; and with token
tiles that divide the pairs, the pairs of a group cover the same row tiles
at the same k-blocks (the W_base reads they share).
"""
import ctypes
import random

import pytest

import bit_weight_delta_gb300 as bd

REC = 10


def schedule(n_pairs, t_total, sk_lo, sk_tiles, n_kb):
    lib = bd.load()
    n = ctypes.c_int64(0)
    assert lib.bitdelta_debug_split_schedule(n_pairs, t_total, sk_lo, sk_tiles, n_kb, None, 0,
                                             ctypes.byref(n)) == 0
    buf = (ctypes.c_int64 * (REC * max(n.value, 1)))()
    assert lib.bitdelta_debug_split_schedule(n_pairs, t_total, sk_lo, sk_tiles, n_kb, buf,
                                             n.value, ctypes.byref(n)) == 0
    return [tuple(buf[REC * i:REC * i + REC]) for i in range(n.value)]


def check(n_pairs, t_total, sk_lo, sk_tiles, n_kb):
    recs = schedule(n_pairs, t_total, sk_lo, sk_tiles, n_kb)
    owner = {}
    by_tile = {}
    slots = set()
    for (pair, tile, kb0, kb1, j, shared, p_lo, p_hi, j_lo, counter) in recs:
        assert sk_lo <= tile < sk_lo + sk_tiles
        assert 0 <= kb0 < kb1 <= n_kb
        for kb in range(kb0, kb1):
            assert (tile, kb) not in owner
            owner[(tile, kb)] = pair
        by_tile.setdefault(tile, []).append((pair, kb0, kb1, j, shared, p_lo, p_hi, j_lo,
                                             counter))
        assert shared == (0 if (kb0, kb1) == (0, n_kb) else 1)
        if shared:
            assert (pair, j) not in slots
            slots.add((pair, j))
    assert len(owner) == sk_tiles * n_kb
    for tile, parts in by_tile.items():
        if len(parts) == 1:
            assert parts[0][4] == 0
            continue
        assert len(parts) == 2, parts
        parts.sort(key=lambda r: r[1])
        lo, hi = parts
        assert lo[2] == hi[1]                          # contiguous in k
        for r in parts:
            assert r[5:7] == (lo[0], hi[0])            # contributors in k order
            assert r[7] == lo[3]                       # the first one's slot
            assert r[8] == tile - sk_lo                # the tile's own counter
        assert hi[3] == 0                              # the second one's range starts here
    return recs


@pytest.mark.parametrize("n_pairs,t_total,sk_lo,sk_tiles,n_kb", [
    (76, 4, 76, 84, 256),      # QKV at M = 2048: a round of whole tiles, then 84 split
    (76, 4, 0, 128, 256),      # O at M = 2048 split whole
    (76, 4, 0, 128, 896),      # down
    (76, 3, 76, 83, 12),       # 3 token tiles: one group
    (76, 1, 0, 81, 32),
    (19, 4, 0, 20, 5),
    (5, 1, 0, 7, 1),
])
def test_split_schedule(n_pairs, t_total, sk_lo, sk_tiles, n_kb):
    check(n_pairs, t_total, sk_lo, sk_tiles, n_kb)


def test_split_schedule_groups_share_w_reads():
    """M = 2048 (4 token tiles), 76 pairs: the pairs of equal index in the
    four groups take the same row tiles at the same k-blocks."""
    recs = schedule(76, 4, 76, 84, 256)
    by_pair = {}
    for r in recs:
        by_pair.setdefault(r[0], []).append(((r[1] - 76) // 4, r[2], r[3]))
    for idx in range(19):
        ref = by_pair[4 * idx]
        for g in range(1, 4):
            assert by_pair[4 * idx + g] == ref


def test_split_schedule_random():
    rng = random.Random(7)
    for _ in range(150):
        t_total = rng.randint(1, 5)
        n_pairs = rng.randint(1, 80)
        sk_tiles = rng.randint(n_pairs, 3 * n_pairs + 3)
        if rng.random() < 0.5:
            sk_tiles = -(-sk_tiles // t_total) * t_total
        sk_lo = t_total * rng.randint(0, 20) + (rng.randint(0, t_total - 1) if rng.random() < 0.2 else 0)
        check(n_pairs, t_total, sk_lo, sk_tiles, rng.randint(1, 40))


def test_split_schedule_rejects():
    lib = bd.load()
    n = ctypes.c_int64(0)
    assert lib.bitdelta_debug_split_schedule(76, 4, 0, 75, 8, None, 0, ctypes.byref(n)) == 1
    assert lib.bitdelta_debug_split_schedule(0, 4, 0, 75, 8, None, 0, ctypes.byref(n)) == 1
    assert lib.bitdelta_debug_split_schedule(4, 4, 0, 8, 8, None, 0, None) == 1
