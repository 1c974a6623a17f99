"""Pins for the CPU oracle: every routine is checked against something other
than itself -- closed forms, library routines (numpy / torch), exhaustive
enumeration and exact rational arithmetic -- so that a dropped term, a wrong
sign or index, a transposed operand or a rounding slip fails here.

The oracle computes the plain definition of C = A x B ("Part 4 -- Pipelining
and Occupancy", section 4.3, the local-sum triple loop); the pipelined
kernels must reach exactly this ("pipeline-gpu-kernel", Step 5: pipelining
only reorders loads)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from software_pipelined_tiled_pipeline_gb300 import synth
from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS

LAYOUTS = ["row_col", "row_row"]


def store_b(Blog: np.ndarray, layout: str) -> np.ndarray:
    """Logical K x N matrix -> storage array for the layout."""
    return np.ascontiguousarray(Blog.T if layout == "row_col" else Blog)


# --------------------------------------------------------------------------
# conversions
# --------------------------------------------------------------------------

def test_f16_decode_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_f16(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_bf16_decode_exhaustive_matches_float32_upper_half():
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.decode_bf16(bits.astype(np.uint16))
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _f16_round_cases(rng):
    xs = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.999, 65520.0, 65536.0, 1e6, -1e6,
          2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12),
          1 + 2 ** -11, 1 + 3 * 2 ** -11, 1 + 2 ** -11 + 2 ** -40, 1 + 2 ** -11 - 2 ** -40,
          float("inf"), float("-inf"), 1e-30, -1e-30]
    xs += list(rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 6, 20000))
    # exact halfway points between neighbouring binary16 values
    h = rng.integers(0, 0x7bff, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    xs += list((lo + hi) / 2)
    return np.array(xs, dtype=np.float64)


def test_round_f16_matches_numpy_correct_rounding():
    # numpy converts float64 -> float16 directly with round-to-nearest-even
    rng = np.random.default_rng(1)
    xs = _f16_round_cases(rng)
    ours = oracle.round_f16(xs)
    ref = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert oracle.round_f16(np.array([np.nan]))[0] & 0x7c00 == 0x7c00


def _bf16_nearest_even_fraction(x: float) -> float:
    """Independent method: walk the bfloat16 grid with exact fractions."""
    if x == 0:
        return 0.0
    s = -1 if x < 0 else 1
    a = Fraction(abs(x))
    # candidate neighbours from all finite positive bfloat16 values near a
    e = Fraction(1)
    exp = 0
    while e * 2 <= a:
        e *= 2
        exp += 1
    while e > a:
        e /= 2
        exp -= 1
    exp = max(exp, -126)
    ulp = Fraction(2) ** (exp - 7)
    q = a / ulp
    fl = q.numerator // q.denominator
    d = q - fl
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * ulp
    maxf = (2 - Fraction(2) ** -7) * Fraction(2) ** 127
    if v > maxf:
        return s * float("inf")
    return s * float(v)


def test_round_bf16_matches_torch_on_float32_values():
    # torch rounds float32 -> bfloat16 to nearest even; float32-exact doubles
    # have no double-rounding issue.
    rng = np.random.default_rng(2)
    x32 = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    ours = oracle.round_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_bf16_matches_exact_fraction_rounding():
    rng = np.random.default_rng(3)
    xs = [1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40, 1 + 2 ** -8 - 2 ** -40, -(1 + 2 ** -8 + 2 ** -45),
          3.0e38, 3.4e38, -3.3e38, 1e-39, 5e-41, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135]
    xs += list(rng.standard_normal(3000) * 10.0 ** rng.integers(-20, 20, 3000))
    xs = np.array(xs, dtype=np.float64)
    ours = oracle.decode_bf16(oracle.round_bf16(xs))
    ref = np.array([_bf16_nearest_even_fraction(float(x)) for x in xs])
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# INT8 -> INT32
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 2, 5), (7, 5, 33), (16, 9, 128), (5, 13, 300)])
def test_i8_all_ones_is_K(layout, M, N, K):
    A = np.ones((M, K), np.int8)
    B = store_b(np.ones((K, N), np.int8), layout)
    assert np.array_equal(oracle.gemm_i8(A, B, layout), np.full((M, N), K, np.int32))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_i8_all_minus_128(layout):
    M, N, K = 4, 6, 517
    A = np.full((M, K), -128, np.int8)
    B = store_b(np.full((K, N), -128, np.int8), layout)
    assert np.array_equal(oracle.gemm_i8(A, B, layout), np.full((M, N), 16384 * K, np.int32))


def test_i8_sum_wraps_modulo_2_32():
    K = 131073                      # 16384 * K exceeds 2^31 - 1
    A = np.full((1, K), -128, np.int8)
    B = np.full((1, K), -128, np.int8)
    expect = 16384 * K - (1 << 32)
    assert oracle.gemm_i8(A, B, "row_col")[0, 0] == expect
    A[0, :2] = 127
    expect2 = (16384 * (K - 2) + 2 * (127 * -128) + (1 << 31)) % (1 << 32) - (1 << 31)
    assert oracle.gemm_i8(A, B, "row_col")[0, 0] == expect2


@pytest.mark.parametrize("layout", LAYOUTS)
def test_i8_identity_and_permutation(layout):
    rng = np.random.default_rng(4)
    K, N = 37, 11
    Blog = rng.integers(-128, 128, (K, N)).astype(np.int8)
    B = store_b(Blog, layout)
    eye = np.eye(K, dtype=np.int8)
    assert np.array_equal(oracle.gemm_i8(eye, B, layout), Blog.astype(np.int32))
    perm = rng.permutation(K)
    P = eye[perm]
    assert np.array_equal(oracle.gemm_i8(P, B, layout), Blog[perm].astype(np.int32))
    # negated identity flips every sign
    assert np.array_equal(oracle.gemm_i8(-eye, B, layout), -Blog.astype(np.int32))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_i8_rank1_outer_product(layout):
    rng = np.random.default_rng(5)
    a = rng.integers(-128, 128, (9, 1)).astype(np.int8)
    b = rng.integers(-128, 128, (1, 14)).astype(np.int8)
    C = oracle.gemm_i8(a, store_b(b, layout), layout)
    assert np.array_equal(C, np.outer(a[:, 0].astype(np.int64), b[0].astype(np.int64)).astype(np.int32))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 4), (7, 5, 33), (33, 17, 129), (64, 40, 1000)])
def test_i8_random_matches_numpy_int64(layout, M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = rng.integers(-128, 128, (M, K)).astype(np.int8)
    Blog = rng.integers(-128, 128, (K, N)).astype(np.int8)
    ref = (A.astype(np.int64) @ Blog.astype(np.int64)).astype(np.int32)
    assert np.array_equal(oracle.gemm_i8(A, store_b(Blog, layout), layout), ref)


def test_i8_transpose_symmetry():
    # (A B)^T = B^T A^T: swapping operands and layouts must transpose C.
    rng = np.random.default_rng(6)
    A = rng.integers(-128, 128, (13, 40)).astype(np.int8)
    Blog = rng.integers(-128, 128, (40, 21)).astype(np.int8)
    C = oracle.gemm_i8(A, store_b(Blog, "row_col"), "row_col")
    Ct = oracle.gemm_i8(np.ascontiguousarray(Blog.T), store_b(A.T, "row_col"), "row_col")
    assert np.array_equal(C.T, Ct)


def test_i8_rows_and_points_agree_with_full():
    A, B = synth.operands("i8", "row_col", 50, 30, 70, seed=9)
    full = oracle.gemm_i8(A, B, "row_col")
    rows = [0, 7, 49, 7]
    assert np.array_equal(oracle.gemm_i8(A, B, "row_col", rows=rows), full[rows])
    r = np.array([0, 3, 49, 10]); c = np.array([0, 29, 5, 10])
    assert np.array_equal(oracle.points_i8(A, B, r, c, "row_col"), full[r, c])


def test_i8_empty_shapes():
    A = np.zeros((0, 5), np.int8)
    B = np.zeros((3, 5), np.int8)
    assert oracle.gemm_i8(A, B).shape == (0, 3)
    A = np.zeros((2, 0), np.int8)
    B = np.zeros((3, 0), np.int8)
    assert np.array_equal(oracle.gemm_i8(A, B), np.zeros((2, 3), np.int32))


# --------------------------------------------------------------------------
# FP16 / BF16 / FP32 inputs
# --------------------------------------------------------------------------

def _as_type(x: np.ndarray, t: str):
    """Values exactly representable in type t -> the oracle's operand form."""
    if t == "f16":
        return x.astype(np.float16)
    if t == "bf16":
        return synth._f32_to_bf16_bits(x.astype(np.float32))
    return x.astype(np.float32)


@pytest.mark.parametrize("t", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_float_integer_valued_inputs_are_exact(t, layout):
    rng = np.random.default_rng(7)
    M, N, K = 19, 23, 150
    hi = 16 if t == "bf16" else 64           # exactly representable integers
    A = rng.integers(-hi, hi + 1, (M, K))
    Blog = rng.integers(-hi, hi + 1, (K, N))
    C = oracle.gemm_ref(_as_type(A, t), store_b(_as_type(Blog, t), layout), t, layout)
    assert np.array_equal(C, (A @ Blog).astype(np.float64))


@pytest.mark.parametrize("t", ["f16", "bf16", "f32"])
def test_float_all_ones_and_rank1(t):
    M, N, K = 6, 10, 77
    A = _as_type(np.ones((M, K)), t)
    B = _as_type(np.ones((N, K)), t)
    assert np.array_equal(oracle.gemm_ref(A, B, t, "row_col"), np.full((M, N), float(K)))
    rng = np.random.default_rng(8)
    a = rng.uniform(-1, 1, (M, 1)); b = rng.uniform(-1, 1, (1, N))
    a_t = _as_type(a, t); b_t = _as_type(b, t)
    av = oracle.decode_bf16(a_t) if t == "bf16" else a_t.astype(np.float64)
    bv = oracle.decode_bf16(b_t) if t == "bf16" else b_t.astype(np.float64)
    C = oracle.gemm_ref(a_t, np.ascontiguousarray(b_t.T), t, "row_col")
    assert np.array_equal(C, np.outer(av[:, 0], bv[0]))


def _exact_product(Av: np.ndarray, Bv: np.ndarray):
    M, K = Av.shape
    N = Bv.shape[1]
    out = [[Fraction(0)] * N for _ in range(M)]
    Af = [[Fraction(float(v)) for v in row] for row in Av]
    Bf = [[Fraction(float(v)) for v in row] for row in Bv]
    for i in range(M):
        for j in range(N):
            out[i][j] = sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0))
    return out


@pytest.mark.parametrize("t", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_float_random_within_double_rounding_of_exact(t, layout):
    rng = np.random.default_rng(11)
    M, N, K = 5, 4, 45
    A = _as_type(rng.uniform(-1, 1, (M, K)), t)
    Blog = _as_type(rng.uniform(-1, 1, (K, N)), t)
    dec = (lambda x: oracle.decode_bf16(x)) if t == "bf16" else (lambda x: x.astype(np.float64))
    Av, Bv = dec(A), dec(Blog)
    exact = _exact_product(Av, Bv)
    C = oracle.gemm_ref(A, store_b(Blog, layout), t, layout)
    absum = np.abs(Av) @ np.abs(Bv)
    bound = K * 2.0 ** -52 * absum              # K roundings of at most 1/2 ulp each
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(float(C[i, j])) - exact[i][j]) <= Fraction(float(bound[i, j]))
    # the float64 library product agrees to the same bound
    assert np.all(np.abs(C - Av @ Bv) <= 2 * bound)


@pytest.mark.parametrize("t", ["f16", "bf16"])
def test_layouts_agree_and_transpose_symmetry_float(t):
    if t == "f16":
        A, B = synth.operands("f16", "row_col", 12, 9, 64, seed=3)
    else:
        A, B = synth.operands("bf16", "row_col", 12, 9, 64, seed=3)
    Blog = np.ascontiguousarray(B.T)             # K x N
    C1 = oracle.gemm_ref(A, B, t, "row_col")
    C2 = oracle.gemm_ref(A, Blog, t, "row_row")
    assert np.array_equal(C1, C2)
    Ct = oracle.gemm_ref(B, np.ascontiguousarray(A), t, "row_col")   # B^T-rows times A^T
    # each entry is the same set of exact products; sums may round in a different
    # order only if the loop order differed -- it does not, so equality is exact.
    assert np.array_equal(C1.T, Ct)


def test_points_and_rows_agree_with_full_float():
    A, B = synth.operands("bf16", "row_col", 40, 24, 96, seed=5)
    full = oracle.gemm_ref(A, B, "bf16", "row_col")
    rows = [39, 0, 5]
    assert np.array_equal(oracle.gemm_ref(A, B, "bf16", "row_col", rows=rows), full[rows])
    r = np.array([1, 39, 20]); c = np.array([23, 0, 11])
    assert np.array_equal(oracle.points_ref(A, B, "bf16", r, c, "row_col"), full[r, c])


def test_f32_loop_exact_on_dyadic_inputs():
    rng = np.random.default_rng(12)
    M, N, K = 8, 8, 64
    A = (rng.integers(-32, 33, (M, K)) / 8.0).astype(np.float32)
    B = (rng.integers(-32, 33, (K, N)) / 4.0).astype(np.float32)
    assert np.array_equal(oracle.gemm_f32_loop(A, B, "row_row").astype(np.float64),
                          oracle.gemm_ref(A, B, "f32", "row_row"))


@pytest.mark.parametrize("wname,rows", [("f32_1024", 16), ("f16_4096", 4), ("bf16_8192_k16384", 2)])
def test_float_loop_error_is_far_inside_the_tolerance(wname, rows):
    # Information line: the plain loop with a float accumulator ("Part 4 -- Pipelining and
    # Occupancy", section 4.3) is what an FP32-accumulating kernel computes in one summation
    # order.  On rows of the workloads' own inputs its error against the exact sum stays far
    # inside the parity tolerance, so the tolerance admits every correct FP32 accumulation
    # order while still being a fraction of max|C|.
    w = WORKLOADS[wname]
    A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    r = list(range(rows))
    ref = oracle.gemm_ref(A, B, w.dtype, w.layout, rows=r)
    # (FP16 operands are numpy half floats, BF16 ones raw bit patterns)
    dec = {"f32": lambda x: x, "f16": lambda x: x.astype(np.float32), "bf16": oracle.decode_bf16}[w.dtype]
    Af = np.asarray(dec(A[:rows]), dtype=np.float32)
    Bf = np.asarray(dec(B), dtype=np.float32)
    loop = oracle.gemm_f32_loop(Af, Bf, w.layout).astype(np.float64)
    err = float(np.max(np.abs(loop - ref)))
    tol = oracle.tolerance(w.K, ref, "f32")
    print("%s: FP32 loop max|err| = %.3g, tolerance %.3g (%.2g of it), max|C| %.3g"
          % (wname, err, tol, err / tol, float(np.max(np.abs(ref)))))
    assert 0 < err < tol / 100
    assert tol < 0.1 * float(np.max(np.abs(ref)))


def test_rounded_output_is_nearest_of_exact():
    # round_f16(C_ref) equals the binary16 value nearest the exact sum when the
    # exact sum is not within double rounding distance of a tie.
    rng = np.random.default_rng(13)
    A = rng.uniform(-1, 1, (6, 40)).astype(np.float16)
    Blog = rng.uniform(-1, 1, (40, 7)).astype(np.float16)
    C = oracle.gemm_ref(A, store_b(Blog, "row_col"), "f16", "row_col")
    got = oracle.round_f16(C).view(np.float16).astype(np.float64)
    exact = _exact_product(A.astype(np.float64), Blog.astype(np.float64))
    for i in range(6):
        for j in range(7):
            e = exact[i][j]
            cand = np.float16(float(e)).astype(np.float64)   # numpy: correctly rounded from double
            assert got[i, j] == cand


def test_tolerance_formula():
    c = np.array([[-3.0, 2.0], [1.0, 0.5]])
    assert oracle.tolerance(256, c) == pytest.approx(0.03)
    assert oracle.tolerance(1024, c) == pytest.approx(0.06)
    assert oracle.tolerance(1024, c, "bf16") == pytest.approx(0.06)
    # below K ~ 39 the stated bound is under one bfloat16 rounding: floored at 2^-8
    assert oracle.tolerance(8, c, "bf16") == pytest.approx(3 * 2.0 ** -8)
    assert oracle.tolerance(8, c, "f16") == pytest.approx(1e-2 * (8 / 256) ** 0.5 * 3)


def test_tolerance_admits_correct_rounding_of_exact_result():
    # a correctly rounded bfloat16 output of the exact sum must always pass
    rng = np.random.default_rng(14)
    for K in (1, 2, 8, 40, 256):
        A = _as_type(rng.uniform(-1, 1, (16, K)), "bf16")
        B = _as_type(rng.uniform(-1, 1, (16, K)), "bf16")
        ref = oracle.gemm_ref(A, B, "bf16", "row_col")
        rounded = oracle.decode_bf16(oracle.round_bf16(ref))
        assert np.max(np.abs(rounded - ref)) <= oracle.tolerance(K, ref, "bf16")
