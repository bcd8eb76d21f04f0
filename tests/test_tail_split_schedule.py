"""The K-chunked tensor kernel's schedule, replayed on the CPU (no GPU).

tf32x3_chunked_kernel (csrc/tf32x3.cu: chunked_plan, piece_of) runs one CTA
per SM.  Whole waves of output tiles come first, tile c + i*G on CTA c.  When
the last wave would leave at least half the SMs idle (or there is less than
one wave), its `tail` tiles are split into split = G // tail K segments (at
most K blocks // 2, so each has two blocks or more): segment j of tail tile
t covers K blocks [j*kblocks//split, (j+1)*kblocks//split) on CTA
j*tail + t, after that CTA's whole tiles, and leaves its sum in partial tile
j*tail + t; tf32x3_fixup_kernel adds partial tiles j = 0, 1, ... of each
tail tile in that order.

The test checks on many plans that every K block of every tile is computed
exactly once, that segments tile each split tile's K range in K order, that
no CTA runs more than one segment, that the fix-up reads exactly the partial
tiles written, and that the workspace holds them.
"""
import random

import pytest


def plan(tiles, kblocks, sms):
    """(G, tiles_dp, tail, split) as chunked_plan."""
    G = min(tiles, sms)
    tail = tiles % sms
    if sms < 2 or tail == 0:
        return G, tiles, 0, 0
    split = min(sms // tail, kblocks // 2)
    if split < 2:
        return G, tiles, 0, 0
    return sms, tiles - tail, tail, split


def pieces(c, G, tiles_dp, tail, split, kblocks):
    """(tile, kb0, kb1, slot or None) of CTA c, in order, as piece_of."""
    out = [(t, 0, kblocks, None) for t in range(c, tiles_dp, G)]
    if c < split * tail:
        j, tl = divmod(c, tail)
        out.append((tiles_dp + tl, j * kblocks // split, (j + 1) * kblocks // split, c))
    return out


def check(tiles, kblocks, sms):
    G, tiles_dp, tail, split = plan(tiles, kblocks, sms)
    covered, written = {}, {}
    for c in range(G):
        ps = pieces(c, G, tiles_dp, tail, split, kblocks)
        assert sum(slot is not None for *_, slot in ps) <= 1
        for t, kb0, kb1, slot in ps:
            assert 0 <= t < tiles and 0 <= kb0 < kb1 <= kblocks
            for kb in range(kb0, kb1):
                assert (t, kb) not in covered, f"block {kb} of tile {t} computed twice"
                covered[(t, kb)] = c
            if slot is not None:
                assert kb1 - kb0 >= 2
                assert slot not in written
                written[slot] = (t, kb0, kb1)
    assert len(covered) == tiles * kblocks, "some K blocks are never computed"
    assert len(written) == split * tail
    assert all(0 <= s < split * tail for s in written)   # within the workspace's partial tiles
    for tl in range(tail):
        nxt = 0
        for j in range(split):   # the fix-up's order
            t, kb0, kb1 = written[j * tail + tl]
            assert t == tiles_dp + tl and kb0 == nxt, "segments out of K order"
            nxt = kb1
        assert nxt == kblocks
    # the tail takes at most 1/split of a tile time; the whole tiles as many waves as they fill
    longest = max(sum(kb1 - kb0 for _, kb0, kb1, _ in pieces(c, G, tiles_dp, tail, split, kblocks))
                  for c in range(G))
    assert longest <= (tiles_dp // G) * kblocks + (-(-kblocks // split) if split else
                                                   (kblocks if tiles % sms else 0))


@pytest.mark.parametrize("tiles,kblocks,sms", [
    (2048, 256, 152),   # 8192 x 8192 x 4096 on 128 x 256 tiles: 13 waves + 72 in halves
    (288, 192, 152),    # 3072^3: 136 tail tiles, no split
    (204, 97, 152),     # 2049 x 3071 x 1537 on 128 x 256 tiles: 1 wave + 52 in halves
    (16, 128, 152),     # 512 x 512 x 4096: 9 segments
    (1, 1024, 152),     # 128 x 128 x 32768: one tile in 152 segments
    (1, 3, 152),        # one tile of 3 K blocks: one segment would be too short
    (76, 2, 152), (77, 100, 152), (152, 10, 152), (304, 10, 152), (5, 2, 4), (3, 7, 8),
])
def test_tail_split_fixed_plans(tiles, kblocks, sms):
    check(tiles, kblocks, sms)


def test_tail_split_random_plans():
    rng = random.Random(11)
    for _ in range(300):
        sms = rng.randrange(2, 200)
        check(rng.randrange(1, 5 * sms), rng.randrange(1, 300), sms)
