"""Shared-memory addressing of the SIMT kernels, checked on the CPU: the
TMA-fed kernel here, the cp.async kernels further down.

csrc/simt_tma.cu reads its operand stages with 16-byte loads:
  * K-major stages ([32][128] floats, as TMA writes an M- or N-contiguous box
    with no swizzle): thread columns a_col..a_col+3 and +64 of row kk (A),
    b_col..b_col+3 and +64 (B);
  * M/N-major stages ([128][32] floats, a K-contiguous box written with the
    128-byte swizzle, 16-byte chunk c of row r stored at chunk c ^ (r % 8)):
    rows (or columns) t + 16 j of the thread, four k per load, at float
    offset t*32 + 16*32*j + 4*(kq ^ (t % 8)).
The thread's place comes from thread_coords (Z-order 4 x 8 lanes, 2 warps
across).  For every thread and load this test checks that the offset the
kernel computes is where the swizzle puts the element it wants, that it stays
inside the stage, and that the eight lanes of each quarter-warp (the unit a
16-byte shared load is served in) touch distinct 16-byte bank groups or the
same address: no bank conflicts.
"""
import pytest

BK, BM, BN, THREADS = 32, 128, 128, 256
STAGE_FLOATS = BK * 128


def thread_coords(tid):
    lane, warp = tid & 31, tid >> 5
    lane_row = (lane & 1) | ((lane >> 4) << 1)
    lane_col = (lane >> 1) & 7
    return 4 * ((warp >> 1) * 4 + lane_row), 4 * ((warp & 1) * 8 + lane_col)


def swizzled_offset(r, k):
    """Float offset of element (row r, k) in a [128][32] box with the 128-byte swizzle."""
    return r * BK + 4 * ((k // 4) ^ (r % 8)) + k % 4


def conflict_free(addrs):
    """addrs: float offsets of one 16-byte load by the 32 lanes."""
    for q in range(4):
        groups = {}
        for a in addrs[8 * q:8 * q + 8]:
            assert a % 4 == 0, "16-byte load not 16-byte aligned"
            groups.setdefault((a // 4) % 8, set()).add(a)
        if any(len(v) > 1 for v in groups.values()):
            return False
    return True


def test_thread_coords_cover_the_tile_once():
    cells = set()
    for tid in range(THREADS):
        a_col, b_col = thread_coords(tid)
        for r in list(range(a_col, a_col + 4)) + list(range(64 + a_col, 68 + a_col)):
            for c in list(range(b_col, b_col + 4)) + list(range(64 + b_col, 68 + b_col)):
                assert (r, c) not in cells
                cells.add((r, c))
    assert len(cells) == BM * BN


def test_mn_major_strided_rows_cover_the_tile_once():
    # the swizzled forms own rows ty + 16 j (A) or columns tx + 16 j (B)
    cells = set()
    for tid in range(THREADS):
        a_col, b_col = thread_coords(tid)
        ty, tx = a_col >> 2, b_col >> 2
        for j in range(8):
            for c in list(range(b_col, b_col + 4)) + list(range(64 + b_col, 68 + b_col)):
                cells.add((ty + 16 * j, c))
    assert len(cells) == BM * BN
    cols = {(tid, (thread_coords(tid)[1] >> 2) + 16 * j) for tid in range(THREADS) for j in range(8)}
    assert {c for _, c in cols} == set(range(BN))


@pytest.mark.parametrize("operand", ["A", "B"])
def test_kmajor_fragment_loads(operand):
    for kk in range(BK):
        for h in range(2):
            addrs = []
            for tid in range(THREADS):
                a_col, b_col = thread_coords(tid)
                col = (a_col if operand == "A" else b_col) + 64 * h
                off = kk * 128 + col
                assert 0 <= off and off + 4 <= STAGE_FLOATS
                addrs.append(off)
            for w in range(THREADS // 32):
                assert conflict_free(addrs[32 * w:32 * w + 32]), (operand, kk, h, w)


@pytest.mark.parametrize("operand", ["A", "B"])
def test_swizzled_fragment_loads(operand):
    for kq in range(BK // 4):
        for j in range(8):
            addrs = []
            for tid in range(THREADS):
                a_col, b_col = thread_coords(tid)
                t = (a_col if operand == "A" else b_col) >> 2
                off = t * BK + j * 16 * BK + 4 * (kq ^ (t & 7))   # the kernel's formula
                r = t + 16 * j
                for e in range(4):   # the four k of the load are elements (r, 4 kq + e)
                    assert off + e == swizzled_offset(r, 4 * kq + e)
                assert 0 <= off and off + 4 <= STAGE_FLOATS
                addrs.append(off)
            for w in range(THREADS // 32):
                assert conflict_free(addrs[32 * w:32 * w + 32]), (operand, kq, j, w)


def test_a_planted_conflict_is_detected():
    # without the XOR the eight rows of a quarter-warp hit the same chunk
    addrs = []
    for tid in range(32):
        a_col, _ = thread_coords(tid)
        t = a_col >> 2
        addrs.append(t * BK + 4 * 0)
    assert not conflict_free(addrs)


# ------------------------------------------------------------ cp.async kernels
#
# csrc/simt_sgemm.cuh keeps both operands K-major ([BK][ROWS] floats) with a
# float4-granular XOR: row kk's column c is stored at c ^ swz(kk),
# swz(kk) = (128 / BK) * (kk >> 2).  Writers: 16-byte cp.async of an M/N-
# contiguous operand (element (mn = 4 mq + e, kk) at kk*ROWS + ((4 mq) ^
# swz(kk)) + e) and, for a K-contiguous operand, the corner turn (thread g of
# the slice holds row g / (BK/4), k quad g % (BK/4), and stores its four
# values one float each to rows kk..kk+3 at column row ^ swz(kk)).  Readers:
# the fragment loads at kk*ROWS + (col ^ swz(kk)), col = a_col (+64) or
# b_col + 64 h.

def swz(kk, bk=BK):
    return (128 // bk) * (kk >> 2)


def cpasync_layout(rows, bk=BK):
    """(k, mn) -> float offset, as the 16-byte cp.async writer places it."""
    where = {}
    for kk in range(bk):
        for mq in range(rows // 4):
            for e in range(4):
                where[(kk, 4 * mq + e)] = kk * rows + ((4 * mq) ^ swz(kk, bk)) + e
    return where


def cornerturn_layout(rows, bk=BK, threads=THREADS):
    """(k, mn) -> float offset, and the per-instruction store addresses of
    the corner turn (r: the thread's vector, e: which of its four floats)."""
    kq_n = bk // 4
    where, stores = {}, {}
    for r in range(bk * rows // (4 * threads)):
        for tid in range(threads):
            g = tid + r * threads
            row, kq = g // kq_n, g % kq_n
            kk = 4 * kq
            col = row ^ swz(kk, bk)
            for e in range(4):
                off = (kk + e) * rows + col
                where[(kk + e, row)] = off
                stores.setdefault((r, e), []).append(off)
    return where, stores


@pytest.mark.parametrize("rows", [128, 256])
def test_cpasync_layout_is_a_permutation_read_back_by_the_fragments(rows):
    where = cpasync_layout(rows)
    assert sorted(where.values()) == list(range(BK * rows))
    nsb = rows // 64
    for kk in range(BK):
        for h in range(nsb):
            addrs = []
            for tid in range(THREADS):
                _, b_col = thread_coords(tid)
                col = b_col + 64 * h
                off = kk * rows + (col ^ swz(kk))
                for e in range(4):
                    assert where[(kk, col + e)] == off + e
                addrs.append(off)
            for w in range(THREADS // 32):
                assert conflict_free(addrs[32 * w:32 * w + 32]), (rows, kk, h, w)


def test_cornerturn_layout_matches_the_reads_and_stores_without_conflicts():
    rows = 128
    where, stores = cornerturn_layout(rows)
    assert where == cpasync_layout(rows), "the two writers disagree on the layout"
    for (r, e), offs in stores.items():
        for w in range(THREADS // 32):
            banks = {}
            for off in offs[32 * w:32 * w + 32]:
                banks.setdefault(off % 32, set()).add(off)
            assert all(len(v) == 1 for v in banks.values()), f"store conflict r={r} e={e} warp={w}"
    # the A fragments (a_col and a_col + 64) read back the corner-turned rows
    for kk in range(BK):
        for h in range(2):
            addrs = []
            for tid in range(THREADS):
                a_col, _ = thread_coords(tid)
                col = a_col + 64 * h
                off = kk * rows + (col ^ swz(kk))
                for e in range(4):
                    assert where[(kk, col + e)] == off + e
                addrs.append(off)
            for w in range(THREADS // 32):
                assert conflict_free(addrs[32 * w:32 * w + 32])


def test_cornerturn_without_swizzle_would_conflict():
    offs = []
    for tid in range(32):
        row, kq = tid // (BK // 4), tid % (BK // 4)
        offs.append((4 * kq) * 128 + row)   # no XOR
    banks = {}
    for off in offs:
        banks.setdefault(off % 32, set()).add(off)
    assert any(len(v) > 1 for v in banks.values())


# ------------------------------------------------------------ other staging tiles

def banks_conflict_free_32bit(offs):
    """One 4-byte shared access by 32 lanes: distinct banks or one address."""
    banks = {}
    for off in offs:
        banks.setdefault(off % 32, set()).add(off)
    return all(len(v) == 1 for v in banks.values())


def test_tensor_epilogue_staging_matches_the_c_map_swizzle():
    # csrc/tf32x3.cu, store_tile_rows: lane r of the warp holds row r of a
    # 32 x 32 fp32 block and writes its 16-byte chunk j to byte
    # r * 128 + ((j ^ (r & 7)) << 4) of a 4 KB buffer, which the TMA store
    # reads through a tensor map with the 128-byte swizzle (chunk c of row r
    # at chunk c ^ (r % 8)).
    for j in range(8):
        offs = []
        for lane in range(32):
            byte = lane * 128 + ((j ^ (lane & 7)) << 4)
            assert byte == lane * 128 + 16 * ((j) ^ (lane % 8))   # the swizzle's definition
            assert 0 <= byte and byte + 16 <= 4096
            offs.append(byte // 4)
        assert conflict_free(offs), j


@pytest.mark.parametrize("rows_in_tile", [32, 64])
def test_padded_transpose_tiles(rows_in_tile):
    # split_transpose (csrc/tf32x3.cu, tile[32][33]) and transpose_kernel
    # (csrc/turn.cu, tile[64][33]): 256 threads as 32 x 8 (tx, ty); writes
    # tile[ty + 8 i][tx], reads tile[tx + 32 (i / 4)][ty + 8 (i % 4)] (the
    # 32-row tile reads tile[tx][ty + 8 i]).
    pitch = 33
    writes, reads = {}, {}
    for tid in range(THREADS):
        tx, ty = tid & 31, tid >> 5
        for i in range(rows_in_tile // 8):
            writes.setdefault(i, {})[tid] = (ty + 8 * i) * pitch + tx
            if rows_in_tile == 64:
                reads.setdefault(i, {})[tid] = (tx + 32 * (i >> 2)) * pitch + ty + 8 * (i & 3)
            else:
                reads.setdefault(i, {})[tid] = tx * pitch + ty + 8 * i
    filled = sorted(o for d in writes.values() for o in d.values())
    assert len(set(filled)) == len(filled) == rows_in_tile * 32
    assert set(o for d in reads.values() for o in d.values()) == set(filled), \
        "the reads do not cover exactly what was written"
    for table in (writes, reads):
        for i, per_tid in table.items():
            for w in range(THREADS // 32):
                assert banks_conflict_free_32bit([per_tid[t] for t in range(32 * w, 32 * w + 32)])


def test_wide_transpose_tiles():
    # split_transpose_wide (csrc/tf32x3.cu) and transpose_vec_kernel
    # (csrc/turn.cu): a 32 x 128 block of X (32 source rows, 128 contiguous
    # columns) through tile[32][129].  Load: thread t takes columns
    # 4 (t % 32) .. +3 of rows t / 32 + 8 i (one 16-byte global load each) and
    # writes them as four floats; store: thread t reads tile[4 (t % 8) + e]
    # [t / 8 + 32 i] for e < 4 and writes them as one 16-byte row segment of
    # the output (4 consecutive source rows of one column).
    pitch = 129
    cells_written, cells_read = [], []
    for i in range(4):
        for e in range(4):
            w_addrs, r_addrs = [], []
            for tid in range(THREADS):
                lr, lk = 4 * (tid & 31), tid >> 5
                row, col = lk + 8 * i, lr + e
                w_addrs.append(row * pitch + col)
                cells_written.append((row, col))
                kq, sr = tid & 7, tid >> 3
                rrow, rcol = 4 * kq + e, sr + 32 * i
                r_addrs.append(rrow * pitch + rcol)
                cells_read.append((rrow, rcol))
            for w in range(THREADS // 32):
                # the tile reads are conflict-free; the scalar writes of a
                # 16-byte load meet at most 4-way conflicts (4 lanes 32 floats
                # apart in the same bank), which the test bounds
                assert banks_conflict_free_32bit(r_addrs[32 * w:32 * w + 32]), (i, e, w)
                banks = {}
                for a in w_addrs[32 * w:32 * w + 32]:
                    banks.setdefault(a % 32, set()).add(a)
                assert max(len(v) for v in banks.values()) <= 4
    full = {(r, c) for r in range(32) for c in range(128)}
    assert len(cells_written) == len(set(cells_written)) and set(cells_written) == full
    assert len(cells_read) == len(set(cells_read)) and set(cells_read) == full


@pytest.mark.parametrize("bn", [128, 256])
def test_tensor_c_store_column_rule(bn):
    # csrc/tf32x3.cu, store_tile_rows / store_running_rows with tma_n: the C
    # map is N rounded down to a multiple of 4 wide (n4); a 32-column block
    # ending at or before tma_n (n4, or no limit when N % 4 == 0) goes through
    # the map, which clips it at n4; the block holding the last columns of a
    # width that is not a multiple of 4 is stored by the threads, up to N.
    # Every column once, no TMA granule past n4 (16 bytes = 4 floats).
    for N in list(range(1, 300)) + [3071, 3072, 2049, 4097]:
        n4 = N // 4 * 4
        tma_n = 1 << 30 if N % 4 == 0 else n4
        seen = []
        for n0 in range(0, N, bn):
            for c in range(bn // 32):
                b0 = n0 + 32 * c
                if b0 >= N:
                    break
                if b0 + 32 <= tma_n:
                    cols = range(b0, min(b0 + 32, n4))
                    assert n4 % 4 == 0 and all(col < n4 for col in cols)
                else:
                    cols = range(b0, min(b0 + 32, N))
                seen.extend(cols)
        assert sorted(seen) == list(range(N)), N
