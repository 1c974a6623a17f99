"""Float parity at full size, and exactness through every scheduling path.

1. The headline launch (FP16 4096^3, the library's default: CTA pairs with a
   stream-K tail) is compared with the oracle on every one of its 16.8 M
   outputs, within the float bound of the parity tests.

2. Integer-valued operands: sparse {-1, 0, +1} entries (the ``ternary``
   distribution of the seeded generator) make every exact sum an integer far
   below 2^8.  FP32 accumulation is then exact in any order, so the FP16/BF16
   output must equal the oracle's exact sum rounded to the output type, bit for
   bit -- on the CTA-pair ring with its stream-K split, on the clusters that
   split 256 x 128 tiles' K-loops in two, on one CTA per tile, and on the
   register-staged baseline.  A K step lost, repeated or added into the wrong
   tile changes some output by at least 1, where the float bound (4 % of
   max|C| at K = 4096) could let it pass.  This is the oracle's exact-integer
   pin ("Part 4 -- Pipelining and Occupancy", section 4.3: the product is the
   plain triple-loop sum) applied to the GPU paths.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import operands, run
from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS

pytestmark = pytest.mark.gpu


def _bits(C: torch.Tensor) -> np.ndarray:
    return C.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_f16_4096_headline_launch_every_element():
    w = WORKLOADS["f16_4096"]
    A, B = operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    C, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=0)
    p = st["plan"]
    assert (p["kernel"], p["cta_pair"]) == ("umma_pair_ring", 1) and p["sk_tiles"] > 0
    ref = oracle.gemm_ref(A, B, w.dtype, w.layout)
    got = C.float().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - ref)))
    assert err <= oracle.tolerance(w.K, ref, w.dtype)
    # an FP32-accumulated, FP16-rounded sum is within about one output rounding of the exact one:
    # far inside the bound (which a lost K step could still meet)
    assert err <= 2.0 ** -10 * float(np.max(np.abs(ref)))


EXACT_CASES = [
    # dtype, M, N, K, launch options, expected plan fields (sk: stream-K split tiles or none)
    ("f16", 4096, 4096, 4096, {}, {"cta_pair": 1, "sk": True}),                # pairs + stream-K tail
    ("bf16", 4096, 4096, 4096, {}, {"cta_pair": 1, "sk": True}),
    ("bf16", 8192, 8192, 4096, {}, {"cta_pair": 1, "sk": True}),               # the BF16 sweep's shape
    ("bf16", 8192, 128, 8192, {}, {"cta_pair": 3}),                            # K split over two pairs
    ("f16", 8192, 128, 8192, {}, {"cta_pair": 3}),
    ("f16", 4096, 4096, 4096, {"no_cta_pair": True}, {"cta_pair": 0, "sk": True}),   # one CTA, stream-K tail
    ("f16", 4096, 4096, 4096, {"one_tile_per_cta": True}, {"persistent": 0}),  # the ring, one tile per CTA
    ("bf16", 1000, 1800, 1040, {}, {"cta_pair": 1, "sk": False}),              # ragged M, N, K, whole tiles
    ("f16", 2056, 776, 4104, {"stages": 3}, {"cta_pair": 1, "sk": True}),      # ragged, every tile split
]


@pytest.mark.parametrize("dtype,M,N,K,opts,plan", EXACT_CASES)
def test_exact_integer_products(dtype, M, N, K, opts, plan):
    A, B = operands(dtype, "row_col", M, N, K, seed=M + N + K, dist="ternary")
    opts = dict(opts)
    stages = opts.pop("stages", 0)
    C, st = run(dtype, "row_col", A, B, M, N, K, variant="pipelined", stages=stages, **opts)
    plan = dict(plan)
    sk = plan.pop("sk", None)
    for k, v in plan.items():
        assert st["plan"][k] == v, (k, st["plan"][k])
    if sk is not None:
        assert (st["plan"]["sk_tiles"] > 0) == sk
    ref = oracle.gemm_ref(A, B, dtype, "row_col")
    assert np.abs(ref).max() < 256 and np.all(ref == np.round(ref))
    want = oracle.round_f16(ref) if dtype == "f16" else oracle.round_bf16(ref)
    got = _bits(C)
    bad = np.argwhere(got != want)
    assert bad.size == 0, "%d outputs differ, first at %s: got %#06x want %#06x" % (
        len(bad), tuple(bad[0]), got[tuple(bad[0])], want[tuple(bad[0])])


@pytest.mark.parametrize("variant", ["pingpong", "nopipe"])
def test_exact_integer_products_register_staged(variant):
    M, N, K = 2048, 2048, 4096
    A, B = operands("f16", "row_col", M, N, K, seed=77, dist="ternary")
    C, _ = run("f16", "row_col", A, B, M, N, K, variant=variant)
    want = oracle.round_f16(oracle.gemm_ref(A, B, "f16", "row_col"))
    assert np.array_equal(_bits(C), want)
