"""Pins for the CPU oracle: each checks it against something other than itself.

The oracle computes C = op(A) op(B) in fp64, ascending k, rounded once to fp32
("CUDA GEMM operator performance optimization", section 1.1; DD2360 workbook,
section 14.3 lab).  The pins below use closed forms (identity, all-ones,
unit selectors, +-1 scale), exact integer products, exact rational brute
force on tiny inputs, a library routine (NumPy float64 matmul) and layout
invariants.  ``test_planted_mistakes_are_caught`` recompiles the oracle with
one plausible bug at a time and checks that some pin fails for every bug.
"""
import os
import shutil
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers that do not use the oracle
# --------------------------------------------------------------------------

def f32_round(q: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) float32 of an exact rational."""
    f = np.float32(float(q))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - q)
        if best is None or d < best[0] or (
                d == best[0] and (int(cand.view(np.uint32)) & 1) == 0):
            best = (d, cand)
    return best[1]


def ulp_diff(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    xi = x.astype(np.float32).view(np.int32).astype(np.int64)
    yi = y.astype(np.float32).view(np.int32).astype(np.int64)
    xi = np.where(xi < 0, -(xi & 0x7FFFFFFF), xi)
    yi = np.where(yi < 0, -(yi & 0x7FFFFFFF), yi)
    return np.abs(xi - yi)


def ops(case):
    return case["opA"][0], case["opB"][0]


# --------------------------------------------------------------------------
# pins: each takes a loaded oracle library and raises AssertionError on failure
# --------------------------------------------------------------------------

def pin_rational_bruteforce(lib):
    """Tiny random problems vs the exact rational sum, correctly rounded."""
    for (M, N, K, seed) in [(2, 2, 2, 1), (3, 3, 3, 2), (2, 3, 5, 3), (4, 1, 7, 4), (1, 5, 1, 5)]:
        c = workloads.make_operands(M, N, K, dist="uniform", seed=seed, key=100)
        a, b = ops(c)
        got = oracle.sgemm(c["A"], c["B"], M, N, K, lib=lib)
        for i in range(M):
            for j in range(N):
                q = sum((Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(K)),
                        Fraction(0))
                assert got[i, j] == f32_round(q), (M, N, K, i, j)


def pin_hand_2x2_3x3(lib):
    """Small integer problems whose products are written out term by term."""
    A = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    want = np.array([[1 * 5 + 2 * 7, 1 * 6 + 2 * 8], [3 * 5 + 4 * 7, 3 * 6 + 4 * 8]], np.float32)
    assert np.array_equal(oracle.sgemm(A, B, 2, 2, 2, lib=lib), want)
    A = np.array([[1, -2, 0], [0, 3, -1], [2, 1, 1]], np.float32)
    B = np.array([[2, 0, 1], [-1, 1, 0], [4, -3, 2]], np.float32)
    want = np.zeros((3, 3), np.float32)
    for i in range(3):
        for j in range(3):
            want[i, j] = A[i, 0] * B[0, j] + A[i, 1] * B[1, j] + A[i, 2] * B[2, j]
    assert np.array_equal(oracle.sgemm(A, B, 3, 3, 3, lib=lib), want)
    # non-square: 2x3 times 3x1
    A = np.array([[1, 2, 3], [-4, 5, -6]], np.float32)
    B = np.array([[7], [8], [9]], np.float32)
    assert np.array_equal(oracle.sgemm(A, B, 2, 1, 3, lib=lib),
                          np.array([[7 + 16 + 27], [-28 + 40 - 54]], np.float32))


def pin_identity(lib):
    """B = I gives C = A bit for bit; A = I gives C = B."""
    c = workloads.make_operands(37, 37, 37, dist="normal", seed=7, key=101)
    a, b = ops(c)
    eye = np.eye(37, dtype=np.float32)
    assert np.array_equal(oracle.sgemm(a, eye, 37, 37, 37, lib=lib), a)
    assert np.array_equal(oracle.sgemm(eye, b, 37, 37, 37, lib=lib), b)


def pin_all_ones(lib):
    """All-ones A (M x K) and B (K x N) give C = K everywhere."""
    for (M, N, K) in [(5, 7, 1), (33, 17, 129), (8, 8, 3000)]:
        A = np.ones((M, K), np.float32)
        B = np.ones((K, N), np.float32)
        assert np.array_equal(oracle.sgemm(A, B, M, N, K, lib=lib), np.full((M, N), K, np.float32))


def pin_unit_selector(lib):
    """A = e_p e_q^T picks row q of B into row p of C, zeros elsewhere."""
    M, N, K = 9, 11, 13
    c = workloads.make_operands(M, N, K, dist="normal", seed=8, key=102)
    _, b = ops(c)
    for (p, q) in [(0, 0), (8, 12), (3, 5)]:
        A = np.zeros((M, K), np.float32)
        A[p, q] = 1.0
        want = np.zeros((M, N), np.float32)
        want[p] = b[q]
        assert np.array_equal(oracle.sgemm(A, b, M, N, K, lib=lib), want)


def pin_integer_exact(lib):
    """Small-integer inputs: every partial sum is an exact float, so C equals
    the exact int64 product bit for bit (including transposed storage)."""
    w = workloads.get("sgemm_256x256x256_int")
    c = workloads.make_case(w)
    a, b = ops(c)
    exact = a.astype(np.int64) @ b.astype(np.int64)
    assert np.array_equal(oracle.sgemm(c["A"], c["B"], 256, 256, 256, lib=lib),
                          exact.astype(np.float32))
    for tA, tB in [(1, 0), (0, 1), (1, 1)]:
        c = workloads.make_operands(70, 45, 133, transA=tA, transB=tB, dist="int",
                                    lda=(72 if tA else 136), ldb=(136 if tB else 48),
                                    poison=True, seed=9, key=103)
        a, b = ops(c)
        exact = (a.astype(np.int64) @ b.astype(np.int64)).astype(np.float32)
        got = oracle.sgemm(c["A"], c["B"], 70, 45, 133, transA=tA, transB=tB,
                           lda=c["lda"], ldb=c["ldb"], lib=lib)
        assert np.array_equal(got, exact), (tA, tB)


def pin_numpy_float64(lib):
    """A library routine: NumPy float64 matmul rounded to float32 agrees to
    within one unit in the last place (only the fp64 summation order differs)."""
    M, N, K = 96, 80, 700
    c = workloads.make_operands(M, N, K, dist="uniform", seed=10, key=104)
    a, b = ops(c)
    ref = (a.astype(np.float64) @ b.astype(np.float64)).astype(np.float32)
    got = oracle.sgemm(c["A"], c["B"], M, N, K, lib=lib)
    d = ulp_diff(got, ref)
    assert d.max() <= 1 and (d == 0).mean() > 0.99


def pin_transpose_storage(lib):
    """The same logical product from transposed storage is bit-identical,
    and NaN-filled padding never reaches the result."""
    M, N, K = 41, 29, 57
    base = None
    for tA in (0, 1):
        for tB in (0, 1):
            c = workloads.make_operands(M, N, K, transA=tA, transB=tB, dist="normal",
                                        lda=(44 if tA else 60), ldb=(60 if tB else 32),
                                        poison=True, seed=11, key=105)
            got = oracle.sgemm(c["A"], c["B"], M, N, K, transA=tA, transB=tB,
                               lda=c["lda"], ldb=c["ldb"], lib=lib)
            assert np.isfinite(got).all()
            if base is None:
                base = got
            assert np.array_equal(got, base), (tA, tB)


def pin_scale_pm1(lib):
    """Entries +-1: the tolerance scale sum|a||b| is exactly K, C has K's parity,
    and |C| <= K."""
    M, N, K = 19, 23, 301
    rng = np.random.default_rng(12)
    A = rng.choice(np.array([-1.0, 1.0], np.float32), size=(M, K)).astype(np.float32)
    B = rng.choice(np.array([-1.0, 1.0], np.float32), size=(K, N)).astype(np.float32)
    C, S = oracle.sgemm(A, B, M, N, K, with_scale=True, lib=lib)
    assert np.array_equal(S, np.full((M, N), float(K)))
    assert np.all(np.abs(C) <= K) and np.all((C.astype(np.int64) - K) % 2 == 0)
    # the scale of 2A and 0.5B is the same K
    _, S2 = oracle.sgemm(2 * A, 0.5 * B, M, N, K, with_scale=True, lib=lib)
    assert np.array_equal(S2, S)


def pin_batched_slices(lib):
    """Batch z of the strided-batched product equals the single product on
    slice z; a zero stride broadcasts one operand."""
    M, N, K, batch = 12, 10, 9, 5
    c = workloads.make_operands(M, N, K, batch=batch, transB=1, dist="normal",
                                sigma=0.125, seed=13, key=106)
    Cb = oracle.sgemm_strided_batched(c["A"], c["B"], M, N, K, batch, transB=1, lib=lib)
    for z in range(batch):
        one = oracle.sgemm(c["A"][z], c["B"][z], M, N, K, transB=1, lib=lib)
        assert np.array_equal(Cb[z], one), z
        exact = (c["opA"][z].astype(np.float64) @ c["opB"][z].astype(np.float64)).astype(np.float32)
        assert ulp_diff(Cb[z], exact).max() <= 1
    Cbb = oracle.sgemm_strided_batched(c["A"], c["B"][0], M, N, K, batch, transB=1,
                                       strideB=0, lib=lib)
    for z in range(batch):
        assert np.array_equal(Cbb[z], oracle.sgemm(c["A"][z], c["B"][0], M, N, K, transB=1, lib=lib))


def pin_entries(lib):
    """Sampled single entries agree with the full product and with closed forms."""
    M, N, K = 31, 27, 65
    for tA, tB in [(0, 0), (1, 1)]:
        c = workloads.make_operands(M, N, K, transA=tA, transB=tB, dist="normal",
                                    seed=14, key=107)
        full, S = oracle.sgemm(c["A"], c["B"], M, N, K, transA=tA, transB=tB,
                               with_scale=True, lib=lib)
        rows = np.array([0, 30, 5, 17, 30])
        cols = np.array([0, 26, 13, 2, 0])
        out, sab = oracle.sgemm_entries(c["A"], c["B"], M, N, K, rows, cols,
                                        transA=tA, transB=tB, lib=lib)
        assert np.array_equal(out, full[rows, cols]) and np.array_equal(sab, S[rows, cols])
    A = np.ones((4, 50), np.float32)
    B = np.ones((50, 3), np.float32)
    out, sab = oracle.sgemm_entries(A, B, 4, 3, 50, [3, 0], [2, 1], lib=lib)
    assert np.array_equal(out, [50, 50]) and np.array_equal(sab, [50, 50])


def pin_degenerate(lib):
    """K = 0 is the empty sum (zeros); M = 0 or N = 0 touch nothing."""
    A = np.zeros((3, 1), np.float32)
    B = np.zeros((1, 4), np.float32)
    C, S = oracle.sgemm(A, B, 3, 4, 0, lda=1, ldb=4, with_scale=True, lib=lib)
    assert np.array_equal(C, np.zeros((3, 4), np.float32)) and not S.any()
    assert oracle.sgemm(A, B, 0, 4, 1, lib=lib).shape == (0, 4)


def pin_ex_reduces_to_plain(lib):
    """alpha = 1, beta = 0, no bias is the plain product bit for bit; alpha = -1
    negates it exactly."""
    M, N, K = 23, 17, 91
    for tA, tB in [(0, 0), (1, 1)]:
        c = workloads.make_operands(M, N, K, transA=tA, transB=tB, dist="normal", seed=16,
                                    key=109)
        plain = oracle.sgemm(c["A"], c["B"], M, N, K, transA=tA, transB=tB, lib=lib)
        ex, _ = oracle.sgemm_ex(c["A"], c["B"], M, N, K, transA=tA, transB=tB, lib=lib)
        assert np.array_equal(ex, plain)
        neg, _ = oracle.sgemm_ex(c["A"], c["B"], M, N, K, alpha=-1.0, transA=tA, transB=tB,
                                 lib=lib)
        assert np.array_equal(neg, -plain)


def pin_ex_integer_closed_form(lib):
    """Integer inputs and integer alpha, beta: alpha*(A@B) + beta*C_in + bias is
    exact, against int64 arithmetic."""
    M, N, K = 31, 29, 57
    c = workloads.make_operands(M, N, K, dist="int", seed=17, key=110)
    a, b = ops(c)
    rng = np.random.default_rng(18)
    C_in = rng.integers(-50, 51, size=(M, N)).astype(np.float32)
    bias = rng.integers(-9, 10, size=N).astype(np.float32)
    for alpha, beta, use_bias in [(3.0, -2.0, True), (0.0, 1.0, True), (-1.0, 0.0, False),
                                  (2.0, 5.0, False), (0.0, 0.0, True)]:
        got, S = oracle.sgemm_ex(c["A"], c["B"], M, N, K, alpha=alpha, beta=beta, C_in=C_in,
                                 bias=bias if use_bias else None, lib=lib)
        want = (int(alpha) * (a.astype(np.int64) @ b.astype(np.int64))
                + int(beta) * C_in.astype(np.int64)
                + (bias.astype(np.int64) if use_bias else 0))
        assert np.array_equal(got, want.astype(np.float32)), (alpha, beta, use_bias)
        scale = (abs(alpha) * (np.abs(a).astype(np.int64) @ np.abs(b).astype(np.int64))
                 + abs(beta) * np.abs(C_in) + (np.abs(bias) if use_bias else 0))
        assert np.array_equal(S, scale.astype(np.float64)), (alpha, beta, use_bias)


def pin_ex_beta_zero_ignores_c_in(lib):
    """beta = 0 never reads C_in: NaN there cannot reach the result."""
    M, N, K = 8, 9, 10
    c = workloads.make_operands(M, N, K, dist="normal", seed=19, key=111)
    nan_c = np.full((M, N), np.nan, np.float32)
    got, _ = oracle.sgemm_ex(c["A"], c["B"], M, N, K, alpha=0.5, beta=0.0, C_in=nan_c,
                             bias=np.ones(N, np.float32), lib=lib)
    assert np.isfinite(got).all()


def pin_ex_rational_bruteforce(lib):
    """Non-dyadic alpha and beta on tiny inputs: the exact rational value,
    correctly rounded."""
    M, N, K = 3, 4, 5
    c = workloads.make_operands(M, N, K, dist="uniform", seed=20, key=112)
    a, b = ops(c)
    rng = np.random.default_rng(21)
    C_in = rng.standard_normal((M, N)).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    alpha, beta = 0.7, -1.3
    got, _ = oracle.sgemm_ex(c["A"], c["B"], M, N, K, alpha=alpha, beta=beta, C_in=C_in,
                             bias=bias, lib=lib)
    for i in range(M):
        for j in range(N):
            dot = sum((Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(K)),
                      Fraction(0))
            q = Fraction(alpha) * dot + Fraction(beta) * Fraction(float(C_in[i, j])) + \
                Fraction(float(bias[j]))
            assert got[i, j] == f32_round(q), (i, j)


PINS = [pin_rational_bruteforce, pin_hand_2x2_3x3, pin_identity, pin_all_ones,
        pin_unit_selector, pin_integer_exact, pin_numpy_float64, pin_transpose_storage,
        pin_scale_pm1, pin_batched_slices, pin_entries, pin_degenerate,
        pin_ex_reduces_to_plain, pin_ex_integer_closed_form, pin_ex_beta_zero_ignores_c_in,
        pin_ex_rational_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.load())


# --------------------------------------------------------------------------
# planted mistakes: every one must be caught by at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "dropped_last_term": ("for (int64_t k = 0; k < j->K; ++k) {\n            const double a = op_a(j, i, k);",
                          "for (int64_t k = 0; k + 1 < j->K; ++k) {\n            const double a = op_a(j, i, k);"),
    "wrong_sign": ("acc[c] += a * op_b(j, k, c);", "acc[c] -= a * op_b(j, k, c);"),
    "transposed_A": ("return j->transA ? (double)j->A[k * j->lda + i] : (double)j->A[i * j->lda + k];",
                     "return j->transA ? (double)j->A[i * j->lda + k] : (double)j->A[k * j->lda + i];"),
    "transposed_B": ("return j->transB ? (double)j->B[c * j->ldb + k] : (double)j->B[k * j->ldb + c];",
                     "return j->transB ? (double)j->B[k * j->ldb + c] : (double)j->B[c * j->ldb + k];"),
    "ignores_ldb": ("(double)j->B[k * j->ldb + c];", "(double)j->B[k * j->N + c];"),
    "float_accumulator": ("double *acc = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));",
                          "float *acc = (float *)calloc((size_t)(N > 0 ? N : 1), sizeof(float));"),
    "scale_without_abs": ("const double aa = fabs(a);", "const double aa = a;"),
    "batch_stride_mixup": ("C + z * strideC, ldc,", "C + z * strideA, ldc,"),
    "entries_off_by_one": ("for (int64_t k = 0; k < K; ++k) {\n            const double a = op_a(&j, i, k), b",
                           "for (int64_t k = 1; k < K; ++k) {\n            const double a = op_a(&j, i, k), b"),
    "row_offset_in_store": ("j->C[i * j->ldc + c] = (float)acc[c];",
                            "j->C[i * j->ldc + (c + 1) % N] = (float)acc[c];"),
    "ex_drops_bias": ("v += (double)bias[c];", "v += 0.0 * (double)bias[c];"),
    "ex_beta_scales_product": ("v += beta * cin;", "v += beta * acc;"),
    "ex_alpha_ignored": ("double v = alpha * acc;", "double v = acc;"),
}


def run_pins_against(lib_path: str) -> list:
    """Names of the pins that fail against the oracle library at lib_path."""
    lib = oracle.load(lib_path)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    # Each mutant runs in a child process: an index mistake can read outside
    # the input buffers, and a crash of the child also counts as caught.
    import subprocess
    import sys
    src = open(oracle.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, f"mut_{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, f"mut_{name}.so")
        oracle.compile_oracle(path, so)
        code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_pins as t; "
                "c = t.run_pins_against(%r); print(c); sys.exit(0 if c else 3)"
                % (os.path.dirname(os.path.dirname(__file__)), os.path.dirname(__file__), so))
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                           timeout=300)
        assert r.returncode != 3, f"no pin catches the planted mistake {name}: {r.stdout}"
        # 0: some pin failed; < 0: the mutant crashed the child (caught too)
        assert r.returncode == 0 or r.returncode < 0, f"mutant runner failed: {r.stderr[-2000:]}"


# --------------------------------------------------------------------------
# closed forms printed on the pages
# --------------------------------------------------------------------------

def _golden_rows():
    rows = []
    for line in open(os.path.join(GOLDEN, "page_figures.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, M, N, K, qty, val, tol, cite = [s.strip() for s in line.split("|")]
        rows.append((name, int(M), int(N), int(K), qty, float(val), float(tol), cite))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_page_figures(row):
    name, M, N, K, qty, val, tol, cite = row
    if qty == "gflop":
        got = workloads.flops(M, N, K) / 1e9
    elif qty == "min_mbytes":
        got = workloads.min_bytes(M, N, K) / 1e6
    elif qty == "flops_e10":
        got = workloads.flops(M, N, K) / 1e10
    elif qty == "naive_read_gb":
        got = 2 * M * N * K * 4 / 1e9
    elif qty == "block_tile_ai":
        got = (M * N * 2 * 8) / ((M * 8 + 8 * N) * 4)   # any BK cancels
    elif qty == "naive_ai":
        got = (2 * K) / (8 * K)
    else:
        raise AssertionError(qty)
    assert abs(got - val) <= tol, (name, got, val, cite)


# --------------------------------------------------------------------------
# the acceptance helpers
# --------------------------------------------------------------------------

def test_tolerance_helpers():
    c = workloads.make_operands(20, 30, 40, dist="normal", seed=15, key=108)
    C, S = oracle.sgemm(c["A"], c["B"], 20, 30, 40, with_scale=True)
    assert oracle.within_tolerance(C, C, S).all()
    bumped = (C.astype(np.float64) + 2e-5 * S + 1e-6).astype(np.float32)
    assert not oracle.within_tolerance(bumped, C, S).any()
    nan = C.copy()
    nan[3, 4] = np.nan
    assert not oracle.within_tolerance(nan, C, S)[3, 4]
    assert oracle.rrmse(C, C) == 0.0
    assert abs(oracle.rrmse((C.astype(np.float64) * 1.001), C) - 0.001) < 1e-9


def test_generator_is_reproducible_and_layout_independent():
    a = workloads.make_operands(33, 21, 17, transA=1, lda=36, poison=True, seed=3, key=5)
    b = workloads.make_operands(33, 21, 17, seed=3, key=5)
    assert np.array_equal(a["opA"], b["opA"]) and np.array_equal(a["opB"], b["opB"])
    assert np.isnan(a["A"][0, :, 33:]).all() and np.array_equal(a["A"][0, :, :33], b["A"][0].T)
    u = workloads.make_operands(64, 64, 64, dist="uniform", seed=0, key=0)["opA"]
    assert u.min() >= -1.0 and u.max() < 1.0
    i = workloads.make_operands(64, 64, 64, dist="int", seed=0, key=0)["opA"]
    assert set(np.unique(i)) <= set(range(-4, 5)) and len(np.unique(i)) == 9
