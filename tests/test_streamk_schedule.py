"""The stream-K schedule's arithmetic, replayed on the CPU (no GPU).

The tile kernels (sgemm_simt_streamk_tma_kernel in csrc/simt_tma.cu,
sgemm_simt_streamk_kernel in csrc/simt_sgemm.cuh) give CTA c of G the units
[c*U/G, (c+1)*U/G) of the U = tiles_sk * kslices K slices of the shared
tiles, as at most two pieces: the tile holding its first unit, and the tile
holding its last.  A piece that is a whole tile is stored to C; any other
goes to workspace slot [c][0] (first piece) or [c][1] (last piece).
streamk_fixup_kernel finds, for each shared tile, the CTAs owning its first
and last slices (streamk_owner) and adds their pieces in CTA order, taking
slot 0 from a CTA whose range starts inside the tile and slot 1 from one
whose range started before it.

The test checks on many plans that every slice of every shared tile is
covered exactly once, that no CTA has more than two pieces, that the fix-up
reads exactly the partial pieces of each tile from the slots they were
written to, in K order, and that whole tiles never reach the fix-up.
"""
import random

import pytest


def owner(u, U, G):
    """The CTA whose range holds unit u (streamk_owner)."""
    return ((u + 1) * G - 1) // U


def pieces_of(c, tiles_sk, kslices, G):
    """(tile, first slice, end slice, slot or None for a whole tile) of CTA c."""
    U = tiles_sk * kslices
    u0, u1 = c * U // G, (c + 1) * U // G
    if u0 == u1:
        return []
    nsk = 1 if u0 // kslices == (u1 - 1) // kslices else 2
    out = []
    for k in range(nsk):
        ub = u0 if k == 0 else (u0 // kslices + 1) * kslices
        tl = ub // kslices
        s0 = ub - tl * kslices
        s1 = min(kslices, s0 + (u1 - ub))
        whole = s0 == 0 and s1 == kslices
        out.append((tl, s0, s1, None if whole else k))
    return out


def fixup_reads(tl, tiles_sk, kslices, G):
    """(CTA, slot) pairs the fix-up adds for shared tile tl, in order, or
    None when one CTA owns the whole tile."""
    U = tiles_sk * kslices
    f, l = tl * kslices, tl * kslices + kslices - 1
    c0, c1 = owner(f, U, G), owner(l, U, G)
    if c0 == c1:
        return None
    reads = []
    for c in range(c0, c1 + 1):
        start = c * U // G
        if (c + 1) * U // G == start:
            continue
        reads.append((c, 0 if start >= f else 1))
    return reads


def check_plan(tiles_sk, kslices, G):
    assert 0 < tiles_sk < G
    covered = {}
    written = {}
    for c in range(G):
        ps = pieces_of(c, tiles_sk, kslices, G)
        assert len(ps) <= 2, f"CTA {c} has {len(ps)} pieces"
        for tl, s0, s1, slot in ps:
            assert 0 <= tl < tiles_sk and 0 <= s0 < s1 <= kslices
            for s in range(s0, s1):
                assert (tl, s) not in covered, f"slice {s} of tile {tl} taken twice"
                covered[(tl, s)] = c
            if slot is not None:
                assert (c, slot) not in written, f"CTA {c} writes slot {slot} twice"
                written[(c, slot)] = (tl, s0, s1)
    assert len(covered) == tiles_sk * kslices, "some slices are never computed"
    read = set()
    for tl in range(tiles_sk):
        reads = fixup_reads(tl, tiles_sk, kslices, G)
        owners = sorted({covered[(tl, s)] for s in range(kslices)})
        if reads is None:
            assert len(owners) == 1
            continue
        assert [c for c, _ in reads] == owners, f"tile {tl}: fix-up reads CTAs {reads}"
        nxt = 0
        for c, slot in reads:
            assert (c, slot) in written, f"tile {tl}: slot {slot} of CTA {c} was never written"
            t, s0, s1 = written[(c, slot)]
            assert t == tl and s0 == nxt, f"tile {tl}: piece {written[(c, slot)]} out of K order"
            nxt = s1
            read.add((c, slot))
        assert nxt == kslices
    assert read == set(written), "a written partial tile is never added"


@pytest.mark.parametrize("tiles_sk,kslices,G", [
    (272, 96, 304),     # 3072^3 on 128 x 128 tiles, two CTAs per SM
    (1, 2, 304), (303, 2, 304), (1, 1000, 304), (151, 48, 152), (7, 3, 8), (2, 2, 3),
    (100, 1, 304),      # a single slice per tile: every piece is a whole tile
])
def test_streamk_schedule_fixed_plans(tiles_sk, kslices, G):
    check_plan(tiles_sk, kslices, G)


def test_streamk_schedule_random_plans():
    rng = random.Random(7)
    for _ in range(400):
        G = rng.randrange(2, 700)
        tiles_sk = rng.randrange(1, G)
        kslices = rng.randrange(1, 160)
        check_plan(tiles_sk, kslices, G)
