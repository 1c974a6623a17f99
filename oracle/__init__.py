"""CPU oracle for the software-pipelined tiled GEMM K-loop.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the C-ABI library and its Python binding) never imports, loads or calls it,
and it imports nothing from the product package.

It wraps ``gemm_oracle.c`` (plain C, built by ``build_oracle.py``), which
computes the plain definition of the product C = A x B -- the local-sum triple
loop of "Part 4 -- Pipelining and Occupancy", section 4.3 "Register reuse":

* INT8 inputs: INT32 sums with two's-complement wrap (the wrap of that
  section's uint32_t loop); exact.
* FP16 / BF16 / FP32 inputs: the stored values converted exactly to double,
  products and sums in double (C_ref); ``round_f16`` / ``round_bf16`` give the
  round-to-nearest-even stored form.

Layouts use the library's names: ``"row_col"`` is A row-major M x K and B
column-major (stored N x K, K contiguous); ``"row_row"`` is A row-major and B
row-major (stored K x N).  Every function accepts an optional list of output
rows (or of (row, col) points) so that full-size problems can be checked on a
sample.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, library routines and exact rational arithmetic.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = build_oracle.build()
    lib = ctypes.CDLL(path)
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_has_openmp.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f64_to_f16_rn.restype = ctypes.c_uint16
    lib.oracle_f64_to_f16_rn.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_bf16_rn.restype = ctypes.c_uint16
    lib.oracle_f64_to_bf16_rn.argtypes = [ctypes.c_double]
    for name in ("oracle_decode_f16", "oracle_decode_bf16", "oracle_round_f16", "oracle_round_bf16"):
        getattr(lib, name).argtypes = [_vp, _vp, _i64]
        getattr(lib, name).restype = None
    lib.oracle_gemm_i8_i32.argtypes = [_vp, _vp, _vp] + [_i64] * 7 + [_vp, _i64]
    lib.oracle_gemm_i8_i32.restype = None
    lib.oracle_gemm_f64.argtypes = [ctypes.c_int, _vp, _vp, _vp] + [_i64] * 7 + [_vp, _i64]
    lib.oracle_gemm_f64.restype = ctypes.c_int
    lib.oracle_gemm_f32_loop.argtypes = [_vp, _vp, _vp] + [_i64] * 7 + [_vp, _i64]
    lib.oracle_gemm_f32_loop.restype = None
    lib.oracle_points_i8_i32.argtypes = [_vp, _vp, _vp] + [_i64] * 5 + [_vp, _vp, _i64]
    lib.oracle_points_i8_i32.restype = None
    lib.oracle_points_f64.argtypes = [ctypes.c_int, _vp, _vp, _vp] + [_i64] * 5 + [_vp, _vp, _i64]
    lib.oracle_points_f64.restype = ctypes.c_int
    _lib = lib
    return lib


_IN_TYPE = {"f16": 0, "bf16": 1, "f32": 2}


def threads() -> int:
    """OpenMP threads the oracle uses (1 without OpenMP)."""
    return _load().oracle_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def has_openmp() -> bool:
    return bool(_load().oracle_has_openmp())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_vp)


def _strides(M, N, K, layout):
    """(a_si, a_sk, b_sk, b_sj) in elements for the named storage layout."""
    if layout == "row_col":
        return K, 1, 1, K          # B stored N x K: B[k][j] at j*K + k
    if layout == "row_row":
        return K, 1, N, 1          # B stored K x N: B[k][j] at k*N + j
    raise ValueError("layout must be 'row_col' or 'row_row'")


def _shape_check(A, B, layout):
    M, K = A.shape
    if layout == "row_col":
        N, K2 = B.shape
    else:
        K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ: A is %s, B is %s (%s)" % (A.shape, B.shape, layout))
    return M, N, K


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    return r, int(r.size)


def _bits16(x, name):
    """FP16 / BF16 operands are passed as their 16-bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("%s must hold 16-bit patterns (uint16) or float16" % name)
    return x


def gemm_i8(A, B, layout="row_col", rows=None) -> np.ndarray:
    """INT32 C (len(rows) x N, or M x N) of int8 A, B with wrap-around sums."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    M, N, K = _shape_check(A, B, layout)
    r, nrows = _rows_arg(rows, M)
    C = np.zeros((nrows, N), dtype=np.int32)
    if nrows and N:
        _load().oracle_gemm_i8_i32(_ptr(A), _ptr(B), _ptr(C), M, N, K, *_strides(M, N, K, layout),
                                   None if r is None else _ptr(r), nrows)
    return C


def gemm_ref(A, B, in_type, layout="row_col", rows=None) -> np.ndarray:
    """C_ref in float64: sums of exact products of the stored inputs.

    ``in_type`` is "f16" or "bf16" (A, B as uint16 bit patterns, or float16 for
    "f16") or "f32" (float32 arrays)."""
    if in_type == "f32":
        A = np.ascontiguousarray(A, dtype=np.float32)
        B = np.ascontiguousarray(B, dtype=np.float32)
    elif in_type in ("f16", "bf16"):
        A = _bits16(A, "A")
        B = _bits16(B, "B")
    else:
        raise ValueError("in_type must be f16, bf16 or f32")
    M, N, K = _shape_check(A, B, layout)
    r, nrows = _rows_arg(rows, M)
    C = np.zeros((nrows, N), dtype=np.float64)
    if nrows and N:
        rc = _load().oracle_gemm_f64(_IN_TYPE[in_type], _ptr(A), _ptr(B), _ptr(C), M, N, K,
                                     *_strides(M, N, K, layout), None if r is None else _ptr(r), nrows)
        if rc != 0:
            raise RuntimeError("oracle_gemm_f64 failed")
    return C


def gemm_f32_loop(A, B, layout="row_row", rows=None) -> np.ndarray:
    """The section 4.3 loop with a float accumulator (information only)."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    M, N, K = _shape_check(A, B, layout)
    r, nrows = _rows_arg(rows, M)
    C = np.zeros((nrows, N), dtype=np.float32)
    if nrows and N:
        _load().oracle_gemm_f32_loop(_ptr(A), _ptr(B), _ptr(C), M, N, K, *_strides(M, N, K, layout),
                                     None if r is None else _ptr(r), nrows)
    return C


def _points_args(A, B, layout, rows, cols):
    M, N, K = _shape_check(A, B, layout)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    if r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N):
        raise IndexError("point out of range")
    a_si, a_sk, b_sk, b_sj = _strides(M, N, K, layout)
    return K, a_si, a_sk, b_sk, b_sj, r, c


def points_i8(A, B, rows, cols, layout="row_col") -> np.ndarray:
    """INT32 C[rows[p], cols[p]] for each sampled point p."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.int8)
    K, a_si, a_sk, b_sk, b_sj, r, c = _points_args(A, B, layout, rows, cols)
    out = np.zeros(r.size, dtype=np.int32)
    if r.size:
        _load().oracle_points_i8_i32(_ptr(A), _ptr(B), _ptr(out), K, a_si, a_sk, b_sk, b_sj,
                                     _ptr(r), _ptr(c), r.size)
    return out


def points_ref(A, B, in_type, rows, cols, layout="row_col") -> np.ndarray:
    """float64 C_ref[rows[p], cols[p]] for each sampled point p."""
    if in_type == "f32":
        A = np.ascontiguousarray(A, dtype=np.float32)
        B = np.ascontiguousarray(B, dtype=np.float32)
    else:
        A = _bits16(A, "A")
        B = _bits16(B, "B")
    K, a_si, a_sk, b_sk, b_sj, r, c = _points_args(A, B, layout, rows, cols)
    out = np.zeros(r.size, dtype=np.float64)
    if r.size:
        rc = _load().oracle_points_f64(_IN_TYPE[in_type], _ptr(A), _ptr(B), _ptr(out), K,
                                       a_si, a_sk, b_sk, b_sj, _ptr(r), _ptr(c), r.size)
        if rc != 0:
            raise RuntimeError("oracle_points_f64 failed")
    return out


def decode_f16(bits) -> np.ndarray:
    x = np.ascontiguousarray(bits, dtype=np.uint16)
    y = np.empty(x.shape, dtype=np.float64)
    _load().oracle_decode_f16(_ptr(x), _ptr(y), x.size)
    return y


def decode_bf16(bits) -> np.ndarray:
    x = np.ascontiguousarray(bits, dtype=np.uint16)
    y = np.empty(x.shape, dtype=np.float64)
    _load().oracle_decode_bf16(_ptr(x), _ptr(y), x.size)
    return y


def round_f16(x) -> np.ndarray:
    """Round-to-nearest-even of float64 values to binary16; returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_f16(_ptr(x), _ptr(y), x.size)
    return y


def round_bf16(x) -> np.ndarray:
    """Round-to-nearest-even of float64 values to bfloat16; returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_ptr(x), _ptr(y), x.size)
    return y


# unit roundoff of the output formats (round to nearest: |fl(x) - x| <= u |x|)
UNIT_ROUNDOFF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 2.0 ** -24}


def tolerance(K: int, c_ref: np.ndarray, out: str = "f32") -> float:
    """Float acceptance bound: max|C - C_ref| <= max(1e-2 * sqrt(K/256), u_out) * max|C_ref|.

    The first term is the stated bound for FP16/BF16/FP32 results.  For very
    small K it falls below one rounding of the output format itself (BF16 below
    K ~ 39, FP16 below K = 1), which no correctly rounded output can meet; the
    bound is then floored at the output's unit roundoff u_out."""
    m = float(np.max(np.abs(c_ref))) if c_ref.size else 0.0
    return max(1e-2 * (K / 256.0) ** 0.5, UNIT_ROUNDOFF[out]) * m
