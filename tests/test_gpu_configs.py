"""GPU parity at the full sizes of the measured workloads, in the launch
configurations the benchmark times.  INT8 4096^3 and the small configs are
compared with the oracle element by element; the large float configs on
sampled rows and points the oracle computes one by one, plus the
stage/variant invariance (identical bits across ring depths)."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_full, check_sampled, operands, run
from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype in (torch.float16, torch.bfloat16) else t


@pytest.mark.parametrize("name", ["i8_256", "f32_1024"])
def test_small_configs_full_compare(name):
    w = WORKLOADS[name]
    A, B = operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    for variant in w.variants:
        stages = w.stages if variant == "pipelined" else (0,)
        for S in stages:
            C, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant=variant, stages=S)
            check_full(w.dtype, w.layout, A, B, C, w.K)


def test_i8_4096_bit_exact_every_stage_and_variant():
    w = WORKLOADS["i8_4096"]
    A, B = operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    ref, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=4)
    check_full(w.dtype, w.layout, A, B, ref, w.K)           # every element against the oracle
    for S in w.stages:
        C, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S)
        assert torch.equal(C, ref)
    for S in w.stages:
        C, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S, i8_engine="imma")
        assert torch.equal(C, ref)
    for S in (2, 6):
        C, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S,
                    i8_engine="tcgen05_2pass")
        assert st["plan"]["kernel"] == "umma_i8_pair_ring"
        assert torch.equal(C, ref)
    for variant in ("pingpong", "nopipe"):
        C, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant=variant)
        assert torch.equal(C, ref)


def test_f16_4096_sampled_and_stage_invariant():
    w = WORKLOADS["f16_4096"]
    A, B = operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    rows = list(range(0, 4096, 67)) + [4095]
    # TMA ring on CTA pairs at 4 stages: two whole waves, the K-loops of the last 104 tiles split
    C, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=4)
    assert st["plan"]["cta_pair"] == 1 and (st["plan"]["dp_tiles"], st["plan"]["sk_tiles"]) == (152, 104)
    check_sampled(w.dtype, w.layout, A, B, C, w.K, rows=rows, npts=4000, seed=1)
    for S in (2, 3):
        C2, st2 = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S)
        assert st2["plan"]["sk_tiles"] == 104
        assert torch.equal(_bits(C2), _bits(C))
    # 5 and 6 stages (the default) split only the 28 tiles left after three whole waves: the same
    # split at both depths, so the same bits; other tiles' partial sums meet in another order
    C6, st6 = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=6)
    assert (st6["plan"]["dp_tiles"], st6["plan"]["sk_tiles"]) == (228, 28)
    check_sampled(w.dtype, w.layout, A, B, C6, w.K, rows=rows, npts=4000, seed=4)
    C5, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=5)
    assert torch.equal(_bits(C5), _bits(C6))
    # one CTA per tile, whole tiles: every variant and depth runs the same MMA sequence
    ref, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=4, no_stream_k=True,
                  no_cta_pair=True)
    assert st["plan"]["sk_tiles"] == 0 and st["plan"]["cta_pair"] == 0
    check_sampled(w.dtype, w.layout, A, B, ref, w.K, rows=rows, npts=4000, seed=2)
    for S in w.stages:
        C2, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S, no_stream_k=True,
                    no_cta_pair=True)
        assert torch.equal(_bits(C2), _bits(ref))
    for variant in ("pingpong", "nopipe"):
        C2, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant=variant)
        assert torch.equal(_bits(C2), _bits(ref))
    # stream-K split of the last wave: differs only by the order of FP32 partial sums
    C3, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=4, no_cta_pair=True)
    assert st["plan"]["sk_tiles"] > 0
    check_sampled(w.dtype, w.layout, A, B, C3, w.K, rows=rows, npts=4000, seed=3)
    for other in (C, C3, C6):
        diff = (other.float() - ref.float()).abs().max().item()
        assert diff <= 2.0 ** -6 * ref.float().abs().max().item()


@pytest.mark.parametrize("name", ["bf16_8192_k256", "bf16_8192_k1024", "bf16_8192_k4096", "bf16_8192_k16384",
                                  "bf16_skinny"])
def test_bf16_sweep_configs(name):
    w = WORKLOADS[name]
    A, B = operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    rows = [0, 1, 127, 128, 4095, 8191] if w.K > 4096 else list(range(0, w.M, 257)) + [w.M - 1]
    ref = None
    for S in w.stages:
        # default launch (stream-K where the tiles do not fill whole waves): sampled oracle check
        C, st = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S)
        check_sampled(w.dtype, w.layout, A, B, C, w.K, npts=1000, seed=S)
        # one CTA per tile, whole tiles: bit-identical across depths
        C2, _ = run(w.dtype, w.layout, A, B, w.M, w.N, w.K, variant="pipelined", stages=S, no_stream_k=True,
                    no_cta_pair=True)
        if ref is None:
            check_sampled(w.dtype, w.layout, A, B, C2, w.K, rows=rows, npts=2000, seed=S)
            ref = C2
        assert torch.equal(_bits(C2), _bits(ref)), "stage %d differs" % S
