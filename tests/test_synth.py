"""The seeded input generator (shared by the CUDA path and the oracle)."""
import numpy as np

from software_pipelined_tiled_pipeline_gb300 import synth


def test_splitmix64_published_first_output():
    # splitmix64 started from state 0 returns 0xE220A8397B1DCDAF first.
    z = synth._mix(np.array([synth.GAMMA], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_draws_are_counter_based():
    a = synth.draws(7, 1, 0, 100)
    b = synth.draws(7, 1, 40, 20)
    assert np.array_equal(a[40:60], b)
    assert not np.array_equal(synth.draws(7, 0, 0, 100), a)
    assert not np.array_equal(synth.draws(8, 1, 0, 100), a)


def test_int8_range_and_determinism():
    A, B = synth.operands("i8", "row_col", 64, 32, 256, seed=1)
    A2, _ = synth.operands("i8", "row_col", 64, 32, 256, seed=1)
    assert A.dtype == np.int8 and A.shape == (64, 256) and B.shape == (32, 256)
    assert np.array_equal(A, A2)
    assert A.min() == -128 and A.max() == 127


def test_uniform_range():
    A, B = synth.operands("f32", "row_row", 128, 64, 100, seed=2)
    assert B.shape == (100, 64)
    assert A.min() >= -1.0 and A.max() < 1.0
    assert abs(float(A.mean())) < 0.02
    H, _ = synth.operands("f16", "row_col", 128, 64, 100, seed=2)
    assert H.dtype == np.float16 and np.all(np.abs(H.astype(np.float32)) <= 1.0)


def test_normal_scaled_moments():
    K = 1024
    A, _ = synth.operands("bf16", "row_col", 256, 8, K, seed=3)
    v = (A.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(v.mean()) < 3e-3
    assert abs(v.std() * np.sqrt(K) - 1.0) < 0.02


def test_chunked_fill_matches_single_draw():
    old = synth._CHUNK
    try:
        synth._CHUNK = 7
        a = synth.int8_uniform(5, 0, (3, 11))
    finally:
        synth._CHUNK = old
    assert np.array_equal(a, synth.int8_uniform(5, 0, (3, 11)))


def test_ternary_values_frequencies_and_encodings():
    A, B = synth.operands("f16", "row_col", 512, 256, 1024, seed=4, dist="ternary")
    v = A.astype(np.float64)
    assert set(np.unique(v)) <= {-1.0, 0.0, 1.0}
    n = v.size
    for val in (1.0, -1.0):   # P = 1/16 each: within 5 standard deviations
        assert abs((v == val).sum() - n / 16) < 5 * np.sqrt(n / 16)
    # every float type holds the same integers exactly; int8 gives the pattern itself
    Ab, _ = synth.operands("bf16", "row_col", 512, 256, 1024, seed=4, dist="ternary")
    assert np.array_equal((Ab.astype(np.uint32) << 16).view(np.float32).astype(np.float64), v)
    Af, _ = synth.operands("f32", "row_col", 512, 256, 1024, seed=4, dist="ternary")
    Ai, _ = synth.operands("i8", "row_col", 512, 256, 1024, seed=4, dist="ternary")
    assert np.array_equal(Af.astype(np.float64), v) and np.array_equal(Ai.astype(np.float64), v)
    # same draws as the int8 stream of the same seed: the top 4 bits decide
    d = synth.draws(4, 0, 0, 64) >> np.uint64(60)
    expect = np.where(d == 0, 1, np.where(d == 1, -1, 0))
    assert np.array_equal(Ai.reshape(-1)[:64], expect)
