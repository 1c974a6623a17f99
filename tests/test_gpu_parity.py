"""GPU parity: the CUDA kernels, called through the C ABI, against the CPU
oracle, element by element (bit-exact for INT8; max|C - C_ref| <=
1e-2 * sqrt(K/256) * max|C_ref| for FP16/BF16/FP32).

Sizes span several CTA tiles and ragged tails in M, N and K; every variant
(no overlap, register ping-pong, TMA ring) and every ring depth 1..8 is run.
Targeted cases follow the pitfalls of "pipeline-gpu-kernel" (Common pitfalls:
a dropped epilogue loses the last K slab; an off-by-one buffer index swaps
slabs; the loop-count edge cases num_tiles in {1, S-1, S, S+1, 2S+1}; K not a
multiple of BK) and its invariant (Step 5 item 4): pipelining only reorders
loads, so all variants and depths give identical outputs for a fixed MMA
order."""
import numpy as np
import pytest
import torch

import software_pipelined_tiled_pipeline_gb300 as gp
from gpu_helpers import check_full, check_sampled, host_float, operands, run, to_dev

pytestmark = pytest.mark.gpu

LAYOUT = {"i8": "row_col", "f16": "row_col", "bf16": "row_col", "f32": "row_row"}
BK = {"i8": 128, "f16": 64, "bf16": 64, "f32": 8}
SMALL = {
    "i8": [(256, 256, 256), (300, 196, 400), (129, 68, 16), (520, 260, 1040)],
    "f16": [(256, 256, 256), (300, 264, 200), (130, 72, 8), (520, 392, 776)],
    "bf16": [(256, 256, 256), (300, 264, 200), (130, 72, 8), (520, 392, 776)],
    "f32": [(256, 256, 128), (300, 260, 100), (129, 132, 4), (384, 512, 264)],
}
VARIANTS = ["nopipe", "pingpong", "pipelined"]


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "f32"])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("idx", range(4))
def test_small_shapes(dtype, variant, idx):
    M, N, K = SMALL[dtype][idx]
    lay = LAYOUT[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=100 + idx)
    C, st = run(dtype, lay, A, B, M, N, K, variant=variant)
    check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "f32"])
@pytest.mark.parametrize("stages", range(1, 9))
def test_ring_every_depth(dtype, stages):
    M, N, K = SMALL[dtype][3]
    lay = LAYOUT[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=7)
    C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=stages)
    assert st["plan"]["stages"] == stages
    check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype,bn", [("f16", 256), ("f16", 128), ("f16", 64), ("bf16", 256), ("bf16", 64),
                                      ("i8", 128), ("i8", 64)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_every_tile_width(dtype, bn, variant):
    M, N, K = 264, 520, 392 if dtype != "i8" else 384
    lay = LAYOUT[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=11)
    C, st = run(dtype, lay, A, B, M, N, K, variant=variant, bn=bn)
    assert st["plan"]["bn"] == bn
    check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype", ["i8", "f16", "f32"])
@pytest.mark.parametrize("S", [2, 3, 4])
@pytest.mark.parametrize("nt_of", ["1", "S-1", "S", "S+1", "2S+1"])
def test_k_tile_counts_around_depth(dtype, S, nt_of):
    nt = {"1": 1, "S-1": S - 1, "S": S, "S+1": S + 1, "2S+1": 2 * S + 1}[nt_of]
    if nt < 1:
        pytest.skip("no K tiles")
    lay = LAYOUT[dtype]
    M, N, K = 192, 136, nt * BK[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=nt)
    C, _ = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S)
    check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "f32"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_only_last_k_slab_nonzero(dtype, variant):
    # a dropped drain/epilogue would silently lose exactly this slab
    lay = LAYOUT[dtype]
    M, N = 200, 136
    K = 5 * BK[dtype] + {"i8": 16, "f16": 8, "bf16": 8, "f32": 4}[dtype]   # ragged last slab
    A, B = operands(dtype, lay, M, N, K, seed=3)
    last = (K // BK[dtype]) * BK[dtype]
    A = A.copy()
    B = B.copy()
    A[:, :last] = 0
    if lay == "row_col":
        B[:, :last] = 0
    else:
        B[:last, :] = 0
    C, _ = run(dtype, lay, A, B, M, N, K, variant=variant, stages=3 if variant == "pipelined" else 0)
    check_full(dtype, lay, A, B, C, K)
    assert np.any(host_float(C) != 0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_i8_slab_order_is_kept(variant):
    # K slab t of A holds the constant t+1 and B a fixed random slab: any
    # swapped or repeated slab changes C.
    M, N, nt = 128, 128, 9
    K = nt * 128
    A = np.zeros((M, K), np.int8)
    for t in range(nt):
        A[:, t * 128:(t + 1) * 128] = t + 1
    rng = np.random.default_rng(5)
    B = rng.integers(-128, 128, (N, K)).astype(np.int8)
    C, _ = run("i8", "row_col", A, B, M, N, K, variant=variant, stages=4 if variant == "pipelined" else 0)
    check_full("i8", "row_col", A, B, C, K)


@pytest.mark.parametrize("dtype", ["i8", "f16", "bf16", "f32"])
def test_k_zero_gives_zeros(dtype):
    lay = LAYOUT[dtype]
    M, N = 72, 64
    A = np.zeros((M, 0), np.int8 if dtype == "i8" else np.float32)
    tC = torch.full((M, N), 7, dtype=torch.float32 if dtype != "i8" else torch.int32, device="cuda")
    if dtype in ("f16", "bf16"):
        tC = tC.to(torch.float16 if dtype == "f16" else torch.bfloat16)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    gp.gemm_pipelined(dummy, dummy, tC, M, N, 0, dtype, lay, 0, "pipelined", torch.cuda.current_stream())
    assert gp.gemm_stats(sync=True)["status"] == 0
    assert bool((tC.float() == 0).all())
    del A


def test_empty_output_is_not_touched():
    tC = torch.full((4, 8), 3.0, dtype=torch.float16, device="cuda")
    gp.gemm_pipelined(None, None, tC, 0, 8, 64, "f16", "row_col", 0, "pipelined", 0)
    torch.cuda.synchronize()
    assert bool((tC == 3.0).all())


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32", "i8"])
def test_all_variants_and_depths_bitwise_identical(dtype):
    # pipelining only reorders loads: with the same MMA sequence the outputs agree bit for bit
    # (whole K-loops: where a K-loop is split over CTAs, the variants may cut it at different
    # K steps -- the FP32 ring takes 16 K steps per slot, the register-staged kernels 8)
    lay = LAYOUT[dtype]
    M, N, K = 264, 392, 520 if dtype != "i8" else 512
    A, B = operands(dtype, lay, M, N, K, seed=21)
    ref, st = run(dtype, lay, A, B, M, N, K, variant="nopipe", no_stream_k=True)
    assert st["plan"]["k_splits"] <= 1 and st["plan"]["sk_tiles"] == 0
    check_full(dtype, lay, A, B, ref, K)
    outs = [run(dtype, lay, A, B, M, N, K, variant="pingpong", no_stream_k=True)[0]]
    for S in range(1, 9):
        outs.append(run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True)[0])
    for S in (1, 2, 4):
        # the ring on the ping-pong kernel's launch shape (one CTA per tile)
        o, st1 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, one_tile_per_cta=True)
        assert st1["plan"]["grid"] == st1["plan"]["tiles"] and st1["plan"]["persistent"] == 0
        outs.append(o)
    for o in outs:
        assert torch.equal(o.view(torch.int16) if o.dtype in (torch.float16, torch.bfloat16) else o,
                           ref.view(torch.int16) if ref.dtype in (torch.float16, torch.bfloat16) else ref)


@pytest.mark.parametrize("dtype,M,N,K", [("f16", 2304, 2560, 1032), ("bf16", 1000, 1800, 2056), ("i8", 2048, 3072, 1040)])
def test_raster_group_does_not_change_results(dtype, M, N, K):
    # the tile order is scheduling only: every raster group gives the same output (identical bits with
    # whole tiles; stream-K splits may meet partial sums in another order, within the float bound)
    lay = LAYOUT[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=M + N)
    ref, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", no_stream_k=True)
    check_full(dtype, lay, A, B, ref, K)
    for g in (1, 3, 8, 64):
        C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", no_stream_k=True, raster_gm=g)
        assert st["plan"]["raster_gm"] == g
        assert torch.equal(C.view(torch.int16) if C.dtype != torch.int32 else C,
                           ref.view(torch.int16) if ref.dtype != torch.int32 else ref)
        C, _ = run(dtype, lay, A, B, M, N, K, variant="pipelined", raster_gm=g)
        check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype,M,N,K", [("bf16", 2000, 5000, 192), ("f16", 2048, 4096, 256), ("bf16", 4100, 2000, 128),
                                         ("f16", 1300, 9000, 200)])
def test_b_resident_short_k(dtype, M, N, K):
    # a K-loop that fills the ring: each CTA walks a contiguous run of tiles and keeps the B tile in
    # the ring while the N block repeats (ragged M, N and K edges included); every tile runs the same
    # MMAs in the same order as on the streamed ring, so the bits are the same
    lay = "row_col"
    A, B = operands(dtype, lay, M, N, K, seed=M + K)
    C, st = run(dtype, lay, A, B, M, N, K)
    p = st["plan"]
    assert p["b_resident"] == 1 and p["stages"] == p["k_tiles"] and p["raster_gm"] == -(-M // 128)
    check_full(dtype, lay, A, B, C, K)
    C2, st2 = run(dtype, lay, A, B, M, N, K, raster_gm=8)
    assert st2["plan"]["b_resident"] == 0
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    # back to back on one stream
    C3, _ = run(dtype, lay, A, B, M, N, K)
    assert torch.equal(C.view(torch.int16), C3.view(torch.int16))


def test_repeat_calls_reuse_cached_descriptors():
    A, B = operands("f16", "row_col", 512, 512, 512, seed=2)
    c1, _ = run("f16", "row_col", A, B, 512, 512, 512)
    c2, _ = run("f16", "row_col", A, B, 512, 512, 512)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "i8", "f32"])
def test_lost_load_reports_timeout_and_context_survives(dtype):
    # test hook: the producer skips the final tile load, a consumer's bounded
    # wait runs out, the kernel exits cleanly and the host sees GP_ERR_TIMEOUT
    lay = LAYOUT[dtype]
    M, N, K = 256, 256, 4 * BK[dtype]
    A, B = operands(dtype, lay, M, N, K, seed=1)
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    out = {"i8": torch.int32, "f16": torch.float16, "f32": torch.float32}[dtype]
    tC = torch.empty((M, N), dtype=out, device="cuda")
    gp.gemm_pipelined(tA, tB, tC, M, N, K, dtype, lay, 2, "pipelined", torch.cuda.current_stream(),
                      timeout_ns=20_000_000, inject_lost_load=True)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == gp.GP_ERR_TIMEOUT
    assert st["device_status"] & 0xFF == 1
    # the context is still usable and the status word was cleared
    C, st2 = run(dtype, lay, A, B, M, N, K)
    assert st2["device_status"] == 0
    check_full(dtype, lay, A, B, C, K)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,S", [(1024, 1024, 4096, 4), (1536, 1280, 4096, 3), (1000, 776, 2056, 4),
                                     (2560, 4096, 1536, 2), (520, 392, 8192, 6)])
def test_stream_k_split_tiles(dtype, M, N, K, S):
    # tiles whose K-loops are split across CTAs, partials added by the first-K-step owner
    lay = "row_col"
    A, B = operands(dtype, lay, M, N, K, seed=M + N + K)
    C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_cta_pair=True)
    p = st["plan"]
    assert p["sk_tiles"] > 0 and p["grid"] == st["sm_count"]
    assert p["dp_tiles"] + p["sk_tiles"] == p["tiles"]
    check_full(dtype, lay, A, B, C, K)
    C2, st2 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True, no_cta_pair=True)
    assert st2["plan"]["sk_tiles"] == 0
    diff = (C.float() - C2.float()).abs().max().item()
    assert diff <= 2.0 ** -6 * C2.float().abs().max().item()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_stream_k_split_follows_the_ring_depth(dtype):
    # 99 pair tiles (ragged M, N, K): a ring of 5 or more slots keeps the full wave whole and splits
    # the tiles left over; a ring of at most 4 splits the full wave too.  Both match the oracle, and
    # depths with the same split give the same bits
    lay = "row_col"
    M, N, K = 2800, 2296, 2056
    A, B = operands(dtype, lay, M, N, K, seed=99)
    C6, st6 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=6)
    p6 = st6["plan"]
    G, T = st6["sm_count"] // 2, p6["tiles"]
    assert p6["cta_pair"] == 1 and T == 99 and T > G
    assert (p6["dp_tiles"], p6["sk_tiles"]) == ((T // G) * G, T - (T // G) * G)
    check_full(dtype, lay, A, B, C6, K)
    C5, _ = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=5)
    assert torch.equal(C5.view(torch.int16), C6.view(torch.int16))
    C4, st4 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=4)
    assert (st4["plan"]["dp_tiles"], st4["plan"]["sk_tiles"]) == ((T // G - 1) * G, T - (T // G - 1) * G)
    check_full(dtype, lay, A, B, C4, K)
    C3, _ = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=3)
    assert torch.equal(C3.view(torch.int16), C4.view(torch.int16))


def test_stream_k_repeated_launches_reuse_workspace():
    # flags carry a per-launch epoch: back-to-back launches on one stream stay correct
    A, B = operands("f16", "row_col", 1024, 1024, 4096, seed=9)
    outs = [run("f16", "row_col", A, B, 1024, 1024, 4096, stages=4, no_cta_pair=True)[0] for _ in range(3)]
    check_full("f16", "row_col", A, B, outs[0], 4096)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_stream_k_lost_load_reports_timeout():
    M, N, K = 1024, 1024, 4096
    A, B = operands("f16", "row_col", M, N, K, seed=4)
    tA, tB = to_dev(A, "f16"), to_dev(B, "f16")
    tC = torch.empty((M, N), dtype=torch.float16, device="cuda")
    gp.gemm_pipelined(tA, tB, tC, M, N, K, "f16", "row_col", 4, "pipelined", torch.cuda.current_stream(),
                      timeout_ns=20_000_000, inject_lost_load=True)
    st = gp.gemm_stats(sync=True)
    assert st["plan"]["sk_tiles"] > 0
    assert st["status"] == gp.GP_ERR_TIMEOUT
    C, st2 = run("f16", "row_col", A, B, M, N, K)
    check_full("f16", "row_col", A, B, C, K)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,S", [(256, 256, 320, 1), (200, 264, 264, 2), (384, 520, 1000, 3), (1000, 776, 2056, 4),
                                     (128, 256, 512, 5), (2304, 2560, 640, 6), (4096, 2048, 328, 4)])
def test_cta_pair_kernel(dtype, M, N, K, S):
    # 256 x 256 tile per CTA pair (each CTA 128 rows of A and of B), ragged in M, N, K
    lay = "row_col"
    A, B = operands(dtype, lay, M, N, K, seed=M * 7 + N + K)
    C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S)
    p = st["plan"]
    assert p["cta_pair"] == 1 and p["kernel"] == "umma_pair_ring" and p["grid"] % 2 == 0
    check_full(dtype, lay, A, B, C, K)
    # whole tiles on pairs: the same MMA order as one CTA per tile, bit for bit
    Cd, std = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True)
    assert std["plan"]["cta_pair"] == 1 and std["plan"]["sk_tiles"] == 0
    C1, st1 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True, no_cta_pair=True)
    assert st1["plan"]["cta_pair"] == 0
    assert torch.equal(Cd.view(torch.int16), C1.view(torch.int16))
    if p["sk_tiles"] > 0:
        assert p["grid"] == 2 * (st["sm_count"] // 2) and p["dp_tiles"] + p["sk_tiles"] == p["tiles"]
        diff = (C.float() - Cd.float()).abs().max().item()
        assert diff <= 2.0 ** -6 * Cd.float().abs().max().item()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,S", [(1000, 120, 2056, 5), (520, 128, 1032, 4), (256, 72, 264, 3), (2056, 104, 4104, 5)])
def test_pair_k_split_kernel(dtype, M, N, K, S):
    # each 256 x 128 tile on two CTA pairs, one per half of the K-loop, the halves added through
    # distributed shared memory; ragged in M, N and K (odd numbers of K steps included)
    lay = "row_col"
    A, B = operands(dtype, lay, M, N, K, seed=M + 5 * N + K)
    C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, pair_k_split=1)
    p = st["plan"]
    assert p["cta_pair"] == 3 and p["kernel"] == "umma_pair_ksplit_ring" and p["grid"] % 4 == 0
    check_full(dtype, lay, A, B, C, K)


def test_pair_k_split_full_skinny_and_repeats():
    # the skinny BF16 workload (8192 x 128 x 8192) at full size, sampled, then repeated launches
    M, N, K = 8192, 128, 8192
    A, B = operands("bf16", "row_col", M, N, K, seed=5)
    tA, tB = to_dev(A, "bf16"), to_dev(B, "bf16")
    outs = [torch.empty(M * N, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for C in outs:
        gp.gemm_pipelined(tA, tB, C, M, N, K, "bf16", "row_col", 0, "pipelined", torch.cuda.current_stream(),
                          pair_k_split=1)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["device_status"] == 0 and st["plan"]["cta_pair"] == 3
    check_sampled("bf16", "row_col", A, B, outs[0].view(M, N).cpu(), K, rows=[0, 1, 255, 256, 4095, M - 1],
                  npts=2000, seed=3)
    for C in outs[1:]:
        assert torch.equal(C, outs[0])


@pytest.mark.parametrize("dtype,M,N,K", [("f16", 4096, 4096, 4096), ("bf16", 1000, 1800, 1040), ("f16", 8192, 128, 8192)])
def test_inputs_ready_fp16_bf16_back_to_back(dtype, M, N, K):
    # with the promise, each launch's loads and MMAs start while the previous launch finishes and
    # only its stores wait: results identical to ordinary launches (stream-K and K-split shapes too)
    A, B = operands(dtype, "row_col", M, N, K, seed=M + N + K)
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    ref = torch.empty(M * N, dtype=tdt, device="cuda")
    stream = torch.cuda.current_stream()
    gp.gemm_pipelined(tA, tB, ref, M, N, K, dtype, "row_col", 0, "pipelined", stream)
    outs = [torch.empty(M * N, dtype=tdt, device="cuda") for _ in range(4)]
    for C in outs:
        gp.gemm_pipelined(tA, tB, C, M, N, K, dtype, "row_col", 0, "pipelined", stream, inputs_ready=True)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["device_status"] == 0
    for C in outs:
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    check_sampled(dtype, "row_col", A, B, ref.view(M, N).cpu(), K, rows=[0, 255, 256, M - 1], npts=1500, seed=1)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K,S", [(512, 128, 1024, 8), (1000, 120, 2056, 7), (2304, 1280, 640, 8),
                                     (520, 392, 1032, 7), (4096, 4096, 512, 8)])
def test_cta_pair_128_kernel(dtype, M, N, K, S):
    # 256 x 128 tile per CTA pair (each CTA 128 rows of A, 64 rows of B): 7-8 stages, or N <= 128
    lay = "row_col"
    A, B = operands(dtype, lay, M, N, K, seed=M * 5 + N + K)
    C, st = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S)
    p = st["plan"]
    assert p["cta_pair"] == 1 and (p["bm"], p["bn"]) == (256, 128) and p["grid"] % 2 == 0
    if M * N * K <= 3e9:
        check_full(dtype, lay, A, B, C, K)
    else:
        check_sampled(dtype, lay, A, B, C, K, rows=[0, 1, 255, 256, 2049, M - 1], npts=2000, seed=S)
    # whole tiles on pairs: the same MMA order as one CTA per 128 x 128 tile, bit for bit
    Cd, std = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True)
    assert std["plan"]["cta_pair"] == 1 and std["plan"]["sk_tiles"] == 0
    C1, st1 = run(dtype, lay, A, B, M, N, K, variant="pipelined", stages=4, bn=128, no_stream_k=True)
    assert st1["plan"]["cta_pair"] == 0 and st1["plan"]["bn"] == 128
    assert torch.equal(Cd.view(torch.int16), C1.view(torch.int16))
    if p["sk_tiles"] > 0:
        diff = (C.float() - Cd.float()).abs().max().item()
        assert diff <= 2.0 ** -6 * Cd.float().abs().max().item()


I8_KERNELS = {"tcgen05_2pass": "umma_i8_pair_ring", "tcgen05_overlap": "umma_i8_overlap_pair_ring",
              "imma": "imma_ring"}


@pytest.mark.parametrize("engine", sorted(I8_KERNELS))
@pytest.mark.parametrize("stages", [1, 2, 4, 6])
def test_int8_engines_every_depth(engine, stages):
    M, N, K = 520, 260, 1040 + 2048
    A, B = operands("i8", "row_col", M, N, K, seed=stages)
    C, st = run("i8", "row_col", A, B, M, N, K, variant="pipelined", stages=stages, i8_engine=engine)
    too_deep = engine == "tcgen05_overlap" and stages == 6   # no room for int8 staging: two-pass runs
    assert st["plan"]["kernel"] == I8_KERNELS["tcgen05_2pass" if too_deep else engine]
    check_full("i8", "row_col", A, B, C, K)


@pytest.mark.parametrize("engine", ["tcgen05_2pass", "tcgen05_overlap"])
@pytest.mark.parametrize("K", [16, 1008, 1024, 1040, 2048, 4096, 5136])
@pytest.mark.parametrize("fill", [(-128, -128), (-128, 127), (127, 127)])
def test_int8_tcgen05_exact_at_extremes(engine, K, fill):
    # every product at the int8 extremes: |partial sums| reach 2^24 inside one
    # 1024-element chunk of K and 2^26+ across chunks -- still bit-exact
    M, N = 300, 136
    A = np.full((M, K), fill[0], np.int8)
    B = np.full((N, K), fill[1], np.int8)
    A[::7, : K // 3] = 3
    C, st = run("i8", "row_col", A, B, M, N, K, variant="pipelined", i8_engine=engine)
    assert st["plan"]["kernel"] == I8_KERNELS[engine]
    check_full("i8", "row_col", A, B, C, K)


@pytest.mark.parametrize("M,N,K", [(1280, 4096, 528), (1240, 3976, 528), (4096, 4096, 1024)])
def test_int8_half_tiles_in_the_last_wave(M, N, K):
    # when the whole 256 x 256 tiles leave a last wave at most half full, those tiles run as
    # two 256 x 128 halves on two pairs: exact, and identical to the IMMA engine's result
    A, B = operands("i8", "row_col", M, N, K, seed=M + N + K)
    C, st = run("i8", "row_col", A, B, M, N, K, variant="pipelined", i8_engine="tcgen05_2pass")
    p = st["plan"]
    W = p["grid"] // 2
    r = p["tiles"] % W
    expect = r if (p["tiles"] > W and 0 < 2 * r <= W) else 0
    assert p["kernel"] == "umma_i8_pair_ring" and p["sk_tiles"] == 0
    assert p["half_tiles"] == expect and p["dp_tiles"] == p["tiles"] - expect
    if M * N * K <= 3e9:
        check_full("i8", "row_col", A, B, C, K)
    else:
        check_sampled("i8", "row_col", A, B, C, K, rows=[0, 1, 255, 256, 2049, M - 1], npts=3000, seed=K)
    C2, st2 = run("i8", "row_col", A, B, M, N, K, variant="pipelined", i8_engine="imma")
    assert torch.equal(C, C2)


def test_int8_inputs_ready_pipelines_successive_calls():
    # with the promise that A and B are in place, each call converts its operands while the
    # previous call's GEMM still runs, alternating between two copy buffers; ordinary calls,
    # changes of shape and an FP16 GEMM in between must not disturb it
    shapes = [(1024, 768, 2048), (520, 260, 3088), (2048, 2048, 1024), (256, 4096, 64), (1024, 768, 2048)] * 2
    ready = [True, True, False, True, True, True, True, False, True, True]
    ops = [operands("i8", "row_col", M, N, K, seed=100 + i) for i, (M, N, K) in enumerate(shapes)]
    tens = [(to_dev(A, "i8"), to_dev(B, "i8")) for A, B in ops]
    outs = [torch.empty(M * N, dtype=torch.int32, device="cuda") for M, N, K in shapes]
    Mf, Nf, Kf = 1024, 1024, 2048
    Af, Bf = operands("f16", "row_col", Mf, Nf, Kf, seed=99)
    tAf, tBf = to_dev(Af, "f16"), to_dev(Bf, "f16")
    Cf = torch.empty(Mf * Nf, dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for i, ((M, N, K), (tA, tB), C, r) in enumerate(zip(shapes, tens, outs, ready)):
        if i == 5:
            gp.gemm_pipelined(tAf, tBf, Cf, Mf, Nf, Kf, "f16", "row_col", 0, "pipelined", stream)
        gp.gemm_pipelined(tA, tB, C, M, N, K, "i8", "row_col", 0, "pipelined", stream, inputs_ready=r)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["device_status"] == 0
    for (M, N, K), (A, B), C in zip(shapes, ops, outs):
        check_full("i8", "row_col", A, B, C.view(M, N).cpu(), K)
    check_sampled("f16", "row_col", Af, Bf, Cf.view(Mf, Nf).cpu(), Kf, rows=[0, 511, Mf - 1], npts=2000, seed=7)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (1000, 3000, 2000), (256, 256, 16), (4104, 264, 1040)])
def test_int8_overlapped_conversion_matches_two_pass(M, N, K):
    # the same FP16 MMAs in the same order on the same exact values: identical int32 results
    A, B = operands("i8", "row_col", M, N, K, seed=M ^ N ^ K)
    C2, st2 = run("i8", "row_col", A, B, M, N, K, variant="pipelined", i8_engine="tcgen05_2pass",
                  no_stream_k=True)
    C3, st3 = run("i8", "row_col", A, B, M, N, K, variant="pipelined", i8_engine="tcgen05_overlap")
    assert st3["plan"]["kernel"] == "umma_i8_overlap_pair_ring" and st3["plan"]["sk_tiles"] == 0
    assert torch.equal(C2, C3)

    if M * N * K <= 3e9:
        check_full("i8", "row_col", A, B, C3, K)
    else:
        check_sampled("i8", "row_col", A, B, C3, K, rows=[0, 1, 255, 256, M - 1], npts=2000, seed=K)


def test_int8_overlap_back_to_back_and_shape_changes():
    # launches queued back to back on one stream share the copies and counters: the
    # batch counter alternates between two words and every K-step count is epoch-tagged
    shapes = [(1024, 768, 2048), (520, 260, 3088), (1024, 768, 2048), (256, 4096, 64)] * 3
    ops = [operands("i8", "row_col", M, N, K, seed=i) for i, (M, N, K) in enumerate(shapes)]
    tens = [(to_dev(A, "i8"), to_dev(B, "i8")) for A, B in ops]
    outs = [torch.empty(M * N, dtype=torch.int32, device="cuda") for M, N, K in shapes]
    for (M, N, K), (tA, tB), C in zip(shapes, tens, outs):
        gp.gemm_pipelined(tA, tB, C, M, N, K, "i8", "row_col", 0, "pipelined", torch.cuda.current_stream(),
                          i8_engine="tcgen05_overlap")
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["device_status"] == 0
    for (M, N, K), (A, B), C in zip(shapes, ops, outs):
        check_full("i8", "row_col", A, B, C.view(M, N).cpu(), K)


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 1024), (500, 372, 1000), (256, 128, 4104), (130, 260, 2052)])
def test_ffma_split_k_every_variant(M, N, K):
    # at most half as many 128 x 128 tiles as SMs: the tiles' K-loops are dealt out as equal
    # ranges (one per SM, or fewer for short K-loops); a shared tile's partials are added in K
    # order, the same in every variant
    A, B = operands("f32", "row_row", M, N, K, seed=M + 3 * N + K)
    C, st = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3)
    p = st["plan"]
    units = -(-K // 32) * p["tiles"]
    assert p["k_splits"] >= 2 and p["grid"] == min(st["sm_count"], units // 8) > p["tiles"]
    check_full("f32", "row_row", A, B, C, K)
    for variant, S in (("pipelined", 2), ("pipelined", 8), ("pingpong", 0), ("nopipe", 0)):
        C2, st2 = run("f32", "row_row", A, B, M, N, K, variant=variant, stages=S)
        assert st2["plan"]["k_splits"] == p["k_splits"]
        assert torch.equal(C2, C), (variant, S)


@pytest.mark.parametrize("tile", [(4, 8), (8, 4), (8, 16), (16, 8), (16, 16)])
def test_ffma_thread_tiles_match_the_8x8_bits(tile):
    # every thread tile runs each output's K sum in the same order: identical bits, ragged edges included
    M, N, K = 300, 420, 1000
    A, B = operands("f32", "row_row", M, N, K, seed=77)
    ref, _ = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3)
    check_full("f32", "row_row", A, B, ref, K)
    C, st = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3, ffma_tile=tile)
    assert st["plan"]["kernel"] == "ffma_ring_%dx%d" % tile
    assert st["plan"]["threads"] == (128 // tile[0]) * (128 // tile[1]) + 32
    assert torch.equal(C, ref)


def test_ffma_ranges_over_part_empty_waves():
    # 272 tiles (ragged edges) on one CTA per SM: each CTA takes an equal range of the tiles'
    # K-loops, longer than one K-loop, so a tile is shared by at most two CTAs
    M, N, K = 2000, 2100, 520
    A, B = operands("f32", "row_row", M, N, K, seed=41)
    C, st = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3)
    p = st["plan"]
    assert p["tiles"] > st["sm_count"] and p["grid"] == st["sm_count"] and p["k_splits"] == 2
    check_full("f32", "row_row", A, B, C, K)
    for variant, S in (("pipelined", 8), ("pingpong", 0), ("nopipe", 0)):
        C2, _ = run("f32", "row_row", A, B, M, N, K, variant=variant, stages=S)
        assert torch.equal(C2, C), (variant, S)
    # integer-valued operands: every summation order is exact, so the ranges must reproduce
    # the whole-tile result bit for bit (a K unit lost or added twice would not)
    A, B = operands("f32", "row_row", M, N, K, seed=42, dist="ternary")
    C, _ = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3)
    ref, st = run("f32", "row_row", A, B, M, N, K, variant="pipelined", stages=3, one_tile_per_cta=True)
    assert st["plan"]["grid"] == st["plan"]["tiles"]
    assert torch.equal(C, ref)


def test_ffma_short_k_is_not_split():
    A, B = operands("f32", "row_row", 128, 128, 40, seed=5)
    C, st = run("f32", "row_row", A, B, 128, 128, 40, variant="pipelined", stages=3)
    assert st["plan"]["k_splits"] == 1
    check_full("f32", "row_row", A, B, C, 40)


def test_ffma_split_k_lost_load_reports_timeout():
    M, N, K = 512, 512, 2048
    A, B = operands("f32", "row_row", M, N, K, seed=6)
    tA, tB = to_dev(A, "f32"), to_dev(B, "f32")
    tC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    gp.gemm_pipelined(tA, tB, tC, M, N, K, "f32", "row_row", 3, "pipelined", torch.cuda.current_stream(),
                      timeout_ns=20_000_000, inject_lost_load=True)
    st = gp.gemm_stats(sync=True)
    assert st["plan"]["k_splits"] > 1
    assert st["status"] == gp.GP_ERR_TIMEOUT
    C, st2 = run("f32", "row_row", A, B, M, N, K)
    assert st2["device_status"] == 0
    check_full("f32", "row_row", A, B, C, K)


@pytest.mark.parametrize("M,N,K,S", [(1024, 1024, 4096, 4), (1280, 1536, 3136, 6), (1000, 776, 2064, 3),
                                     (768, 2048, 8192, 2)])
def test_int8_tcgen05_stream_k_exact(M, N, K, S):
    # tiles whose K-loops are split across CTA pairs: int32 partials, so the
    # result is bit-identical to whole-tile scheduling
    A, B = operands("i8", "row_col", M, N, K, seed=M + N + K)
    C, st = run("i8", "row_col", A, B, M, N, K, variant="pipelined", stages=S)
    p = st["plan"]
    assert p["kernel"] == "umma_i8_pair_ring" and p["sk_tiles"] > 0
    assert p["dp_tiles"] + p["sk_tiles"] == p["tiles"]
    check_full("i8", "row_col", A, B, C, K)
    C2, st2 = run("i8", "row_col", A, B, M, N, K, variant="pipelined", stages=S, no_stream_k=True)
    assert st2["plan"]["sk_tiles"] == 0
    assert torch.equal(C, C2)


def test_int8_tcgen05_stream_k_repeated_launches():
    # per-launch epochs on the tile counters: back-to-back launches stay exact
    A, B = operands("i8", "row_col", 1024, 1024, 4096, seed=11)
    outs = [run("i8", "row_col", A, B, 1024, 1024, 4096, stages=6)[0] for _ in range(3)]
    check_full("i8", "row_col", A, B, outs[0], 4096)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_int8_tcgen05_sum_wraps_like_int32():
    # 16384 * 131088 exceeds 2^31 - 1: the INT32 result wraps modulo 2^32
    M, N, K = 128, 128, 131088
    A = np.full((M, K), -128, np.int8)
    B = np.full((N, K), -128, np.int8)
    C, st = run("i8", "row_col", A, B, M, N, K, variant="pipelined")
    assert st["plan"]["sk_tiles"] == 1      # the one tile's K-loop is split over every CTA pair
    want = (16384 * K + (1 << 31)) % (1 << 32) - (1 << 31)
    assert int(C[0, 0]) == want and bool((C == want).all())
