"""CPU models of the kernels' mbarrier pipelines (no GPU).

Each model replays, under random interleavings of the roles, the stage,
phase and parity arithmetic the kernels use, with a barrier that behaves as
an mbarrier: a parity wait on phase k passes once the k-th phase has
completed, and is only meaningful while the barrier has completed k or k + 1
phases (one phase behind, it would pass spuriously; one phase ahead, it would
never pass).  The models assert exactly that at every poll, that no stage is
refilled while a reader still needs it, that every reader sees the slice it
expects, and that every interleaving finishes.

  * The TMA-fed SIMT kernels (csrc/simt_tma.cu, tma_mainloop and the
    persistent kernel): one issuing thread inside warp 0, eight warps
    releasing stages through per-warp arrivals on "empty" barriers, and a
    slice counter carried across the pieces (stream-K) or tiles
    (persistent form) of one CTA.
  * The persistent tensor kernel (csrc/tf32x3.cu): TMA producer, MMA issuer
    with tcgen05.commit releases, optional converter warps between "full"
    and the MMAs, and epilogue warps draining one of ACC_BUFS accumulators.
"""
import random

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete a phase."""

    def __init__(self, count, name):
        self.count, self.name = count, name
        self.pending = count
        self.completed = 0

    def arrive(self, n=1):
        assert 0 < n <= self.pending, f"{self.name}: more arrivals than the phase expects"
        self.pending -= n
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count

    def passed(self, k):
        """Poll for the completion of phase k (0-based) with parity k & 1."""
        assert self.completed in (k, k + 1), \
            f"{self.name}: parity wait on phase {k} with {self.completed} phases completed"
        return self.completed == k + 1


def interleave(roles, rng, limit=200000):
    """Runs generator roles in random order until all finish."""
    alive = list(roles)
    steps = 0
    while alive:
        steps += 1
        assert steps < limit, "no progress: the roles wait on one another"
        i = rng.randrange(len(alive))
        try:
            next(alive[i])
        except StopIteration:
            alive.pop(i)


# ------------------------------------------------------------ SIMT TMA kernels

def simt_tma_pieces(pieces, stages, warps, seed):
    """tma_mainloop over a CTA's pieces (each a number of K slices): slice j
    of a piece is the CTA's slice g0 + j, stage g % stages, full-barrier
    parity (g / stages) & 1; thread 0 (in warp 0) issues slice g after every
    warp released slice g - stages (empty parity (g / stages - 1) & 1),
    first stages - 1 slices of a piece on entry, then one after each of its
    own releases."""
    rng = random.Random(seed)
    full = [Barrier(1, f"full{s}") for s in range(stages)]
    empty = [Barrier(warps, f"empty{s}") for s in range(stages)]
    ring = [None] * stages          # slice a stage holds (landed or in flight)
    landed = [False] * stages
    readers = [set() for _ in range(stages)]
    in_flight = []
    seen = [[] for _ in range(warps)]

    def issue(g):
        s = g % stages
        if g >= stages:
            while not empty[s].passed(g // stages - 1):
                yield
        assert not readers[s], "stage refilled while a warp still reads it"
        ring[s], landed[s] = g, False
        readers[s] = set(range(warps))
        in_flight.append(g)

    def tma():
        while True:
            if in_flight:
                g = in_flight.pop(rng.randrange(len(in_flight)))
                landed[g % stages] = True
                full[g % stages].arrive()
            yield

    def warp(w):
        gk = 0
        for n in pieces:
            g0 = gk
            if w == 0:
                for j in range(min(stages - 1, n)):
                    yield from issue(g0 + j)
            for kt in range(n):
                s = gk % stages
                while not full[s].passed(gk // stages):
                    yield
                assert ring[s] == gk and landed[s], "a warp read the wrong slice"
                seen[w].append(gk)
                gk += 1
                yield
                readers[s].discard(w)
                empty[s].arrive()
                if w == 0 and kt + stages - 1 < n:
                    yield from issue(g0 + kt + stages - 1)

    t = tma()
    roles = [warp(w) for w in range(warps)]
    # the copy engine runs until the warps finish
    def driver():
        alive = list(roles)
        steps = 0
        while alive:
            steps += 1
            assert steps < 500000, "no progress: the roles wait on one another"
            if rng.random() < 0.3:
                next(t)
                continue
            i = rng.randrange(len(alive))
            try:
                next(alive[i])
            except StopIteration:
                alive.pop(i)
    driver()
    total = sum(pieces)
    for w in range(warps):
        assert seen[w] == list(range(total)), f"warp {w} consumed {seen[w]}"
    assert not in_flight, "a copy was issued past the last slice"


@pytest.mark.parametrize("pieces", [[96], [1], [2], [3], [5, 7], [1, 1], [2, 96], [95, 1],
                                    [4, 4, 4, 4]])
def test_simt_tma_pipeline(pieces):
    # 3 stages as the kernels use; 2 and 4 as a check of the arithmetic
    for stages in (3, 2, 4):
        for seed in range(12):
            simt_tma_pieces(pieces, stages, warps=8, seed=seed)


def simt_tma_persistent(tiles, ktiles, stages, warps, seed):
    """The persistent form: one slice counter g over the CTA's tiles x
    ktiles; thread 0 keeps stages - 1 slices ahead across tile boundaries
    (issue g + stages - 1 after releasing g)."""
    pieces_total = tiles * ktiles
    rng = random.Random(seed)
    full = [Barrier(1, f"full{s}") for s in range(stages)]
    empty = [Barrier(warps, f"empty{s}") for s in range(stages)]
    ring = [None] * stages
    readers = [set() for _ in range(stages)]
    in_flight, landed = [], [False] * stages
    seen = [[] for _ in range(warps)]

    def issue(g):
        s = g % stages
        if g >= stages:
            while not empty[s].passed(g // stages - 1):
                yield
        assert not readers[s]
        ring[s], landed[s] = g, False
        readers[s] = set(range(warps))
        in_flight.append(g)

    def warp(w):
        if w == 0:
            for g in range(min(stages - 1, pieces_total)):
                yield from issue(g)
        g = 0
        for _ in range(tiles):
            for _ in range(ktiles):
                s = g % stages
                while not full[s].passed(g // stages):
                    yield
                assert ring[s] == g and landed[s]
                seen[w].append(g)
                yield
                readers[s].discard(w)
                empty[s].arrive()
                if w == 0 and g + stages - 1 < pieces_total:
                    yield from issue(g + stages - 1)
                g += 1
            yield   # the tile's store

    roles = [warp(w) for w in range(warps)]
    alive = list(roles)
    steps = 0
    while alive:
        steps += 1
        assert steps < 500000, "no progress"
        if in_flight and rng.random() < 0.3:
            g = in_flight.pop(rng.randrange(len(in_flight)))
            landed[g % stages] = True
            full[g % stages].arrive()
            continue
        i = rng.randrange(len(alive))
        try:
            next(alive[i])
        except StopIteration:
            alive.pop(i)
    for w in range(warps):
        assert seen[w] == list(range(pieces_total))


def simt_tma_abort(pieces, stages, warps, seed, abort_step):
    """tma_mainloop with the abort path: at step `abort_step` some wait runs
    out and sets the CTA's abort word.  From then on every wait returns at
    once.  A warp releases a stage only if its "full" wait saw the copy land;
    thread 0 refills a stage only once all warps released it (its "empty"
    wait gives up once the word is set, unless the release had already
    completed, so a slice may be skipped and a later one still issued), and
    finish_abort waits for the latest copy issued into each stage.  Checks
    that no stage ever gets a second fill while its previous copy is in
    flight, and that no copy is in flight when the CTA exits."""
    rng = random.Random(seed)
    full = [Barrier(1, f"full{s}") for s in range(stages)]
    empty = [Barrier(warps, f"empty{s}") for s in range(stages)]
    flying = [False] * stages
    in_flight = []
    state = {"abort": False, "step": 0}
    last = [None] * stages            # slice last issued into each stage

    def wait(bar, k):
        # bounded wait: gives up once the abort word is set
        while True:
            if bar.completed == k + 1:
                return True
            if state["abort"]:
                return False
            assert bar.completed == k, f"{bar.name}: parity wait on phase {k} with {bar.completed}"
            yield

    def issue(g):
        s = g % stages
        if g >= stages:
            ok = yield from wait(empty[s], g // stages - 1)
            if not ok:
                return
        assert not flying[s], "a stage got a second fill while its copy was in flight"
        flying[s] = True
        in_flight.append(g)
        last[s] = g

    def tma():
        while True:
            if in_flight:
                g = in_flight.pop(rng.randrange(len(in_flight)))
                flying[g % stages] = False
                full[g % stages].arrive()
            yield

    def warp(w):
        gk = 0
        for n in pieces:
            g0 = gk
            if w == 0:
                for j in range(min(stages - 1, n)):
                    yield from issue(g0 + j)
            for kt in range(n):
                s = gk % stages
                landed = yield from wait(full[s], gk // stages)
                gk += 1
                yield
                if landed:
                    empty[s].arrive()
                if w == 0 and kt + stages - 1 < n:
                    yield from issue(g0 + kt + stages - 1)
        if w == 0 and state["abort"]:
            # finish_abort: the latest fill of every stage lands before exit
            for s in range(stages):
                if last[s] is not None:
                    while full[s].completed < last[s] // stages + 1:
                        yield

    t = tma()
    alive = [warp(w) for w in range(warps)]
    steps = 0
    while alive:
        steps += 1
        assert steps < 500000, "no progress: the roles wait on one another"
        if steps == abort_step:
            state["abort"] = True
        if rng.random() < 0.3:
            next(t)
            continue
        i = rng.randrange(len(alive))
        try:
            next(alive[i])
        except StopIteration:
            alive.pop(i)
    assert state["abort"] or steps < abort_step
    assert not in_flight, "a copy was still in flight when the CTA exited"


@pytest.mark.parametrize("pieces", [[96], [3], [5, 7], [2, 96]])
def test_simt_tma_abort_path(pieces):
    # the abort word set at many points of the run, 3 stages as the kernels use
    for stages in (3, 2):
        for seed in range(40):
            abort_step = random.Random(1000 + seed).randrange(1, 400)
            simt_tma_abort(pieces, stages, warps=8, seed=seed, abort_step=abort_step)


@pytest.mark.parametrize("tiles,ktiles", [(6, 2), (1, 8), (5, 1), (3, 7)])
def test_simt_tma_persistent_pipeline(tiles, ktiles):
    for seed in range(12):
        simt_tma_persistent(tiles, ktiles, stages=3, warps=8, seed=seed)


# ------------------------------------------------------------ tensor kernel

def tensor_persistent(nlocal, kblocks, stages, acc_bufs, conv, seed):
    """tf32x3_persistent_kernel: slice g = i * kblocks + kb in stage
    g % stages.  Producer: waits empty (parity (g / stages - 1) & 1) for
    g >= stages, then the copies complete "full".  Converters (if conv):
    wait full, fill the stage's planes, arrive on "converted" (one arrival
    per converter warp).  MMA: waits acce of its buffer (parity
    (i / acc_bufs - 1) & 1) before tile i >= acc_bufs, then per slice the
    converted (or full) barrier, issues, and commits to empty; after the
    tile, commits to accf.  Commits complete in issue order, after the MMAs.
    Epilogue warps (4) wait accf (parity (i / acc_bufs) & 1), drain, arrive
    on acce."""
    rng = random.Random(seed)
    conv_warps = 4
    full = [Barrier(1, f"full{s}") for s in range(stages)]
    empty = [Barrier(1, f"empty{s}") for s in range(stages)]
    convd = [Barrier(conv_warps, f"conv{s}") for s in range(stages)]
    accf = [Barrier(1, f"accf{b}") for b in range(acc_bufs)]
    acce = [Barrier(4, f"acce{b}") for b in range(acc_bufs)]
    ring = [None] * stages            # (slice, landed, converted warps, consumed)
    acc = [None] * acc_bufs           # (tile, slices accumulated)
    in_flight, commits = [], []
    drained = []
    ready = convd if conv else full

    def producer():
        for i in range(nlocal):
            for kb in range(kblocks):
                g = i * kblocks + kb
                s = g % stages
                if g >= stages:
                    while not empty[s].passed(g // stages - 1):
                        yield
                assert ring[s] is None or ring[s]["consumed"], "stage refilled before its MMAs completed"
                ring[s] = {"g": g, "landed": False, "conv": 0, "consumed": False}
                in_flight.append(g)
                yield

    def converter(w):
        for i in range(nlocal):
            for kb in range(kblocks):
                g = i * kblocks + kb
                s = g % stages
                while not full[s].passed(g // stages):
                    yield
                assert ring[s]["g"] == g and ring[s]["landed"]
                ring[s]["conv"] += 1
                convd[s].arrive()
                yield

    def mma():
        for i in range(nlocal):
            b, u = i % acc_bufs, i // acc_bufs
            if i >= acc_bufs:
                while not acce[b].passed(u - 1):
                    yield
            assert acc[b] is None, "MMAs into an accumulator the epilogue has not drained"
            acc[b] = [i, 0]
            for kb in range(kblocks):
                g = i * kblocks + kb
                s = g % stages
                while not ready[s].passed(g // stages):
                    yield
                st = ring[s]
                assert st["g"] == g and st["landed"] and (not conv or st["conv"] == conv_warps)
                acc[b][1] += 1
                commits.append(("empty", s, g))
                yield
            commits.append(("accf", b, i))

    def epilogue(w):
        for i in range(nlocal):
            b, u = i % acc_bufs, i // acc_bufs
            while not accf[b].passed(u):
                yield
            assert acc[b] == [i, kblocks], f"epilogue read {acc[b]} for tile {i}"
            drained.append((w, i))
            if acce[b].pending == 1:
                acc[b] = None   # the last warp's arrival frees the buffer
            acce[b].arrive()
            yield

    def engines():
        # copies land in any order; commits complete in issue order
        while True:
            r = rng.random()
            if in_flight and r < 0.5:
                g = in_flight.pop(rng.randrange(len(in_flight)))
                ring[g % stages]["landed"] = True
                full[g % stages].arrive()
            elif commits:
                kind, x, n = commits.pop(0)
                if kind == "empty":
                    ring[x]["consumed"] = True
                    empty[x].arrive()
                else:
                    accf[x].arrive()
            yield

    roles = [producer(), mma()] + [epilogue(w) for w in range(4)]
    if conv:
        roles += [converter(w) for w in range(conv_warps)]
    eng = engines()
    alive = list(roles)
    steps = 0
    while alive:
        steps += 1
        assert steps < 500000, "no progress: the roles wait on one another"
        if rng.random() < 0.3:
            next(eng)
            continue
        i = rng.randrange(len(alive))
        try:
            next(alive[i])
        except StopIteration:
            alive.pop(i)
    assert sorted(drained) == sorted((w, i) for w in range(4) for i in range(nlocal))
    assert not in_flight and not commits


@pytest.mark.parametrize("stages,acc_bufs", [(4, 1), (3, 2), (6, 2)])
@pytest.mark.parametrize("conv", [False, True])
@pytest.mark.parametrize("nlocal,kblocks", [(5, 2), (2, 1), (3, 96), (7, 3)])
def test_tensor_persistent_pipeline(stages, acc_bufs, conv, nlocal, kblocks):
    for seed in range(4):
        tensor_persistent(nlocal, kblocks, stages, acc_bufs, conv, seed)


# ------------------------------------------------------------ K-chunked tensor kernel

def piece_chunks(kb0, kb1, kcb):
    """The chunks of a piece of K blocks [kb0, kb1): split at the multiples of
    kcb (tf32x3_chunked_kernel)."""
    return [(max(kb0, c * kcb), min(kb1, (c + 1) * kcb))
            for c in range(kb0 // kcb, (kb1 - 1) // kcb + 1)]


def tensor_chunked(pieces, stages, kcb, seed, nslot=2, epi_warps=8):
    """tf32x3_chunked_kernel: the ring as in the persistent kernel, its fills
    counted across the CTA's pieces (g); piece i = K blocks [kb0, kb1) of a
    tile (a whole tile, or a stream-K piece) splits into chunks at the
    multiples of kcb, and the CTA's chunks, counted across pieces (gc), go to
    chunk accumulator gc % nslot.
    MMA: before chunk gc >= nslot waits "chunk free" of its accumulator
    (parity (gc / nslot - 1) & 1), then per K block the "full" barrier, and
    commits each stage to "empty" and the finished chunk to "chunk full".
    Epilogue warps (8) wait "chunk full" (parity (gc / nslot) & 1), add the
    chunk into their running sums and arrive on "chunk free"; after a piece's
    last chunk they hold the piece's whole sum."""
    rng = random.Random(seed)
    full = [Barrier(1, f"full{s}") for s in range(stages)]
    empty = [Barrier(1, f"empty{s}") for s in range(stages)]
    chf = [Barrier(1, f"chunk_full{s}") for s in range(nslot)]
    che = [Barrier(epi_warps, f"chunk_free{s}") for s in range(nslot)]
    ring = [None] * stages
    acc = [None] * nslot              # [chunk gc, K blocks accumulated]
    in_flight, commits = [], []
    sums = {}                         # (warp, piece) -> K blocks summed

    def producer():
        g = 0
        for kb0, kb1 in pieces:
            for kb in range(kb0, kb1):
                s = g % stages
                if g >= stages:
                    while not empty[s].passed(g // stages - 1):
                        yield
                assert ring[s] is None or ring[s]["consumed"], "stage refilled before its MMAs completed"
                ring[s] = {"g": g, "landed": False, "consumed": False}
                in_flight.append(g)
                g += 1
                yield

    def mma():
        gc = g = 0
        for kb0, kb1 in pieces:
            for c0, c1 in piece_chunks(kb0, kb1, kcb):
                sl, u = gc % nslot, gc // nslot
                if gc >= nslot:
                    while not che[sl].passed(u - 1):
                        yield
                assert acc[sl] is None, "MMAs into a chunk accumulator the epilogue has not drained"
                acc[sl] = [gc, 0]
                for _ in range(c0, c1):
                    s = g % stages
                    while not full[s].passed(g // stages):
                        yield
                    st = ring[s]
                    assert st["g"] == g and st["landed"]
                    acc[sl][1] += 1
                    commits.append(("empty", s, g))
                    g += 1
                    yield
                commits.append(("chf", sl, gc))
                gc += 1

    def epilogue(w):
        gc = 0
        for i, (kb0, kb1) in enumerate(pieces):
            total = 0
            for c0, c1 in piece_chunks(kb0, kb1, kcb):
                sl, u = gc % nslot, gc // nslot
                while not chf[sl].passed(u):
                    yield
                want = c1 - c0
                assert acc[sl] == [gc, want], f"epilogue read {acc[sl]} for chunk {gc}"
                total += acc[sl][1]
                if che[sl].pending == 1:
                    acc[sl] = None   # the last warp's arrival frees the accumulator
                che[sl].arrive()
                gc += 1
                yield
            sums[(w, i)] = total

    def engines():
        while True:
            r = rng.random()
            if in_flight and r < 0.5:
                g = in_flight.pop(rng.randrange(len(in_flight)))
                ring[g % stages]["landed"] = True
                full[g % stages].arrive()
            elif commits:
                kind, x, n = commits.pop(0)
                if kind == "empty":
                    ring[x]["consumed"] = True
                    empty[x].arrive()
                else:
                    chf[x].arrive()
            yield

    roles = [producer(), mma()] + [epilogue(w) for w in range(epi_warps)]
    eng = engines()
    alive = list(roles)
    steps = 0
    while alive:
        steps += 1
        assert steps < 2000000, "no progress: the roles wait on one another"
        if rng.random() < 0.3:
            next(eng)
            continue
        i = rng.randrange(len(alive))
        try:
            next(alive[i])
        except StopIteration:
            alive.pop(i)
    assert sums == {(w, i): kb1 - kb0 for w in range(epi_warps)
                    for i, (kb0, kb1) in enumerate(pieces)}
    assert not in_flight and not commits


@pytest.mark.parametrize("stages,kcb", [(4, 4), (3, 2)])   # the 256- and 128-wide tiles
@pytest.mark.parametrize("nlocal,kblocks", [(2, 9), (3, 8), (1, 1), (4, 3), (2, 193)])
def test_tensor_chunked_pipeline(stages, kcb, nlocal, kblocks):
    for seed in range(4):
        tensor_chunked([(0, kblocks)] * nlocal, stages, kcb, seed)


# Pieces of other lengths: whole tiles followed by a K segment of a tail tile
# that starts and ends inside a chunk, and sequences of segments (one-block
# chunks at either end included).
@pytest.mark.parametrize("stages,kcb", [(4, 4), (3, 2)])
@pytest.mark.parametrize("pieces", [[(0, 9), (0, 9), (5, 9), (0, 2)], [(0, 8), (7, 8), (0, 1)],
                                    [(3, 10)], [(0, 97), (33, 66)], [(1, 2), (0, 5)]])
def test_tensor_chunked_pipeline_segments(stages, kcb, pieces):
    for seed in range(4):
        tensor_chunked(pieces, stages, kcb, seed)
