"""gemm_pipelined_noalloc: the FP16/BF16 TMA-ring GEMM with no device memory
allocation.

Some callers cannot allocate device memory while they run -- a framework that
owns all device memory through its own pool, a serving loop that cannot
afford the device-wide synchronisation of cudaMalloc, a process with a memory
budget fixed at start-up.  For them this entry point takes the stream-K
scratch from a fixed array compiled into the library instead of a workspace
allocated on first use.  These checks call it through the C ABI on shapes whose
plans split K-loops (so the scratch is really used), compare each of two calls
in a row with gemm_pipelined's output within the float tolerance of the parity
tests, and check that the free device memory does not move.

The file is named to be collected last, so a run that stops at the first
failure has run every other test before this one."""
import numpy as np
import pytest
import torch

import oracle
import software_pipelined_tiled_pipeline_gb300 as gp
from gpu_helpers import check_sampled, host_float, operands, to_dev

pytestmark = pytest.mark.gpu

OUT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1024, 1024, 4096), (4096, 4096, 4096), (1000, 776, 2056)])
def test_noalloc_matches_gemm_pipelined_on_two_calls(dtype, M, N, K):
    A, B = operands(dtype, "row_col", M, N, K, seed=M + K)
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    stream = torch.cuda.current_stream()

    ref = torch.empty((M, N), dtype=OUT[dtype], device="cuda")
    gp.gemm_pipelined(tA, tB, ref, M, N, K, dtype, "row_col", 0, "pipelined", stream)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0
    ref_plan = st["plan"]

    outs = [torch.full((M, N), float("nan"), dtype=OUT[dtype], device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for C in outs:
        gp.gemm_pipelined_noalloc(tA, tB, C, M, N, K, dtype, 0, stream)
        st = gp.gemm_stats(sync=True)
        assert st["status"] == 0, gp.strerror(st["status"])
        assert st["plan"]["sk_tiles"] > 0                 # the split path, i.e. the scratch, was used
        assert st["plan"]["sk_tiles"] == ref_plan["sk_tiles"] and st["plan"]["grid"] == ref_plan["grid"]
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_before - free_after < (8 << 20), "device memory was allocated"

    r = host_float(ref.cpu())
    tol = oracle.tolerance(K, r, dtype)
    for C in outs:
        got = host_float(C.cpu())
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - r))) <= tol
    # and against the oracle on sampled points
    check_sampled(dtype, "row_col", A, B, outs[1].cpu(), K, npts=500, seed=3)


def test_noalloc_rejects_other_types_and_handles_empty():
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    assert gp.gemm_pipelined_noalloc(dummy, dummy, dummy, 8, 8, 16, "i8", check=False) == gp.GP_ERR_UNSUPPORTED
    assert gp.gemm_pipelined_noalloc(dummy, dummy, dummy, 8, 8, 16, "f32", check=False) == gp.GP_ERR_UNSUPPORTED
    assert gp.gemm_pipelined_noalloc(None, None, None, 0, 8, 16, "f16", check=False) == gp.GP_OK


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_noalloc_exact_integer_products(dtype):
    # integer-valued operands (sparse -1/0/+1): the exact sums are small integers, so the output
    # must equal the oracle's exact sum rounded to the output type, bit for bit, on the split path
    M, N, K = 4096, 4096, 4096
    A, B = operands(dtype, "row_col", M, N, K, seed=5, dist="ternary")
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    C = torch.full((M, N), float("nan"), dtype=OUT[dtype], device="cuda")
    gp.gemm_pipelined_noalloc(tA, tB, C, M, N, K, dtype, 0, torch.cuda.current_stream())
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["plan"]["sk_tiles"] > 0
    ref = oracle.gemm_ref(A, B, dtype, "row_col")
    want = oracle.round_f16(ref) if dtype == "f16" else oracle.round_bf16(ref)
    got = C.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_noalloc_short_k_keeps_b_in_the_ring(dtype):
    # K = 192 (3 K steps): one CTA per 128 x 256 tile with B kept in the ring; no workspace at all,
    # and the same bits as the allocating entry point
    M, N, K = 2048, 4096, 192
    A, B = operands(dtype, "row_col", M, N, K, seed=11)
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    stream = torch.cuda.current_stream()
    ref = torch.empty((M, N), dtype=OUT[dtype], device="cuda")
    gp.gemm_pipelined(tA, tB, ref, M, N, K, dtype, "row_col", 0, "pipelined", stream)
    assert gp.gemm_stats(sync=True)["status"] == 0
    C = torch.full((M, N), float("nan"), dtype=OUT[dtype], device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    gp.gemm_pipelined_noalloc(tA, tB, C, M, N, K, dtype, 0, stream)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0
    assert st["plan"]["b_resident"] == 1 and st["plan"]["sk_tiles"] == 0 and st["plan"]["stages"] == 3
    assert torch.cuda.mem_get_info()[0] >= free_before - (8 << 20)
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    check_sampled(dtype, "row_col", A, B, C.cpu(), K, npts=500, seed=4)
