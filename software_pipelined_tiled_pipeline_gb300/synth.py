"""Seeded synthetic operands for the GEMM library.

This module holds only the random-number generation that feeds both the CUDA
path and the CPU oracle; it contains none of the product's arithmetic.

Generator: splitmix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), counter-based.  A stream is
identified by (seed, tensor_id); its key is ``mix(2*seed + tensor_id)`` and
its i-th draw is ``mix(key + (i+1)*GAMMA)`` with GAMMA = 0x9E3779B97F4A7C15
and ``mix`` the splitmix64 finaliser.  Draw i feeds the element at flat index
i of the operand in its storage order (A: M x K row-major; B: N x K for the
K-major "row_col" layout, K x N for "row_row").

Distributions (the value ranges of the synthetic square GEMM workloads):

* ``int8``      -- top 8 bits of the draw, uniform on [-128, 127].
* ``uniform``   -- u = (draw >> 40) * 2^-24, value 2u - 1 in [-1, 1), exact in
  float32; float16 operands take its round-to-nearest-even binary16 value.
* ``normal``    -- Box-Muller on draws 2i and 2i+1: u1 = ((d >> 11) + 1) * 2^-53,
  u2 = (d >> 11) * 2^-53, z = sqrt(-2 ln u1) cos(2 pi u2), scaled by 1/sqrt(K),
  rounded to float32 and then to bfloat16 (both round-to-nearest-even).
* ``ternary``   -- sparse integers: +1 if the top 4 bits of the draw are 0, -1
  if they are 1, else 0 (P(+1) = P(-1) = 1/16); exact in every float type.
  A product of two such operands has integer entries far below 2^8 at the
  sizes used here, so its rounded value is the exact sum.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> np.uint64:
    s = np.array([(2 * int(seed) + int(tensor_id)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return _mix(s)[0]


def draws(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the (seed, tensor_id) stream, as uint64."""
    key = stream_key(seed, tensor_id)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    return _mix(key + idx * GAMMA)


def _fill(n, fn, dtype, seed, tensor_id):
    """Generate in chunks of draws (several threads: numpy releases the GIL)."""
    out = np.empty(n, dtype=dtype)
    starts = list(range(0, n, _CHUNK))

    def work(s):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(seed, tensor_id, s, c)

    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1, 16)) as ex:
            list(ex.map(work, starts))
    return out


def _int8_chunk(seed, tid, s, c):
    return (draws(seed, tid, s, c) >> np.uint64(56)).astype(np.uint8).view(np.int8)


def _uniform_chunk(seed, tid, s, c):
    u = (draws(seed, tid, s, c) >> np.uint64(40)).astype(np.float64) * 2.0 ** -24
    return (2.0 * u - 1.0).astype(np.float32)


def int8_uniform(seed: int, tensor_id: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return _fill(n, _int8_chunk, np.int8, seed, tensor_id).reshape(shape)


def f32_uniform(seed: int, tensor_id: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return _fill(n, _uniform_chunk, np.float32, seed, tensor_id).reshape(shape)


def f16_uniform(seed: int, tensor_id: int, shape) -> np.ndarray:
    return f32_uniform(seed, tensor_id, shape).astype(np.float16)


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (finite inputs)."""
    f = x.astype(np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    return ((f + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_normal(seed: int, tensor_id: int, shape, K: int) -> np.ndarray:
    """N(0,1)/sqrt(K) as bfloat16 bit patterns (uint16)."""
    n = int(np.prod(shape))
    scale = 1.0 / np.sqrt(float(K))

    def chunk(sd, tid, s, c):
        d = draws(sd, tid, 2 * s, 2 * c)
        u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return _f32_to_bf16_bits((z * scale).astype(np.float32))

    return _fill(n, chunk, np.uint16, seed, tensor_id).reshape(shape)


def _ternary_chunk(seed, tid, s, c):
    top = draws(seed, tid, s, c) >> np.uint64(60)
    return np.where(top == 0, 1, np.where(top == 1, -1, 0)).astype(np.int8)


def ternary(seed: int, tensor_id: int, shape) -> np.ndarray:
    """Sparse {-1, 0, +1} as int8."""
    return _fill(int(np.prod(shape)), _ternary_chunk, np.int8, seed, tensor_id).reshape(shape)


def operands(dtype: str, layout: str, M: int, N: int, K: int, seed: int, dist: str = None):
    """(A, B) numpy arrays in storage layout.

    dtype: "i8" | "f16" | "bf16" | "f32".  FP16 operands are float16 arrays,
    BF16 operands are uint16 bit patterns.  ``dist`` overrides the default
    distribution ("int8" for i8, "uniform" for f16/f32, "normal" for bf16)."""
    b_shape = (N, K) if layout == "row_col" else (K, N)
    if layout not in ("row_col", "row_row"):
        raise ValueError("layout must be 'row_col' or 'row_row'")
    if dist is None:
        dist = {"i8": "int8", "f16": "uniform", "f32": "uniform", "bf16": "normal"}[dtype]
    gens = {
        ("i8", "int8"): lambda t, sh: int8_uniform(seed, t, sh),
        ("f32", "uniform"): lambda t, sh: f32_uniform(seed, t, sh),
        ("f16", "uniform"): lambda t, sh: f16_uniform(seed, t, sh),
        ("bf16", "normal"): lambda t, sh: bf16_normal(seed, t, sh, K),
        ("bf16", "uniform"): lambda t, sh: _f32_to_bf16_bits(f32_uniform(seed, t, sh)),
        ("f16", "ternary"): lambda t, sh: ternary(seed, t, sh).astype(np.float16),
        ("bf16", "ternary"): lambda t, sh: _f32_to_bf16_bits(ternary(seed, t, sh).astype(np.float32)),
        ("f32", "ternary"): lambda t, sh: ternary(seed, t, sh).astype(np.float32),
        ("i8", "ternary"): lambda t, sh: ternary(seed, t, sh),
    }
    fn = gens.get((dtype, dist))
    if fn is None:
        raise ValueError("no generator for dtype=%s dist=%s" % (dtype, dist))
    return fn(0, (M, K)), fn(1, b_shape)
