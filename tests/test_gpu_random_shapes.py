"""Seeded random shapes through every variant and dtype, each compared element
by element with the oracle: M, N, K drawn across tile and K-step boundaries
(ragged tails, fewer K steps than ring slots, more tiles than SMs), ring depth
and the launch options drawn too.  Alignment rules of the C ABI: K a multiple
of 16 for INT8 and 8 for FP16/BF16 (16-byte rows); N a multiple of 4 for FP32
and 8 otherwise (C and B rows)."""
import numpy as np
import pytest

from gpu_helpers import check_full, operands, run

pytestmark = pytest.mark.gpu

LAYOUT = {"i8": "row_col", "f16": "row_col", "bf16": "row_col", "f32": "row_row"}
K_ALIGN = {"i8": 16, "f16": 8, "bf16": 8, "f32": 4}
N_ALIGN = {"i8": 8, "f16": 8, "bf16": 8, "f32": 4}


def _cases(dtype, n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 90)) * N_ALIGN[dtype]
        K = int(rng.integers(1, 200)) * K_ALIGN[dtype]
        variant = ["pipelined", "pipelined", "pingpong", "nopipe"][int(rng.integers(0, 4))]
        S = int(rng.integers(1, 9)) if variant == "pipelined" else 0
        opts = {}
        if dtype in ("f16", "bf16") and variant == "pipelined":
            opts = [{}, {"no_stream_k": True}, {"no_cta_pair": True}, {"one_tile_per_cta": True}][int(rng.integers(0, 4))]
        if dtype == "i8" and variant == "pipelined" and rng.integers(0, 2):
            opts = [{"i8_engine": "imma"}, {"one_tile_per_cta": True}][int(rng.integers(0, 2))]
        if dtype == "f32" and variant == "pipelined" and rng.integers(0, 2):
            opts = {"ffma_tile": [(4, 8), (8, 4), (8, 16), (16, 8)][int(rng.integers(0, 4))]}
        out.append((M, N, K, variant, S, opts))
    return out


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "f32"])
@pytest.mark.parametrize("batch", range(3))
def test_random_shapes_match_the_oracle(dtype, batch):
    for (M, N, K, variant, S, opts) in _cases(dtype, 8, 1000 * batch + len(dtype)):
        A, B = operands(dtype, LAYOUT[dtype], M, N, K, seed=M * 31 + N * 7 + K)
        C, st = run(dtype, LAYOUT[dtype], A, B, M, N, K, variant=variant, stages=S, **opts)
        check_full(dtype, LAYOUT[dtype], A, B, C, K)
