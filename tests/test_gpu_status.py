"""Per-call status records and the workspace lifecycle, on the GPU.

A bounded wait that gives up is reported only to the call it belongs to:
gemm_stats(sync=1) reads that call's own status slot on that call's stream, so
a timeout on one stream is neither reported to nor cleared by a caller on
another stream.  gemm_release frees the library's workspaces; more than the
tracked number of streams reuse the least recently used workspace."""
import threading

import pytest
import torch

import software_pipelined_tiled_pipeline_gb300 as gp
from gpu_helpers import check_full, operands, to_dev

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_to_its_own_thread_only():
    # thread 1: a call whose last tile load is withheld (its wait gives up after 50 ms);
    # thread 2: a clean call on another stream, whose record is read after thread 1's kernel has
    # finished and before thread 1 reads its own
    M, N, K = 512, 512, 1024
    A, B = operands("f16", "row_col", M, N, K, seed=31)
    tA, tB = to_dev(A, "f16"), to_dev(B, "f16")
    C1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C2 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    k1_done, t2_read = threading.Event(), threading.Event()
    res = {}

    def t1():
        try:
            gp.gemm_pipelined(tA, tB, C1, M, N, K, "f16", "row_col", 2, "pipelined", s1, timeout_ns=50_000_000,
                              inject_lost_load=True)
            s1.synchronize()
            k1_done.set()
            t2_read.wait(60)
            res["t1"] = gp.gemm_stats(sync=True)
        except Exception as e:  # surfaced by the assertions below
            st = gp.gemm_stats(sync=False)
            res["t1_err"] = "%r cuda_error %d at %s, plan %s" % (e, st["cuda_error"],
                                                            gp._binding.SITES.get(st["cuda_error_site"]),
                                                            {k: st["plan"][k] for k in ("kernel", "smem_bytes", "grid")})
            k1_done.set()

    def t2():
        try:
            gp.gemm_pipelined(tA, tB, C2, M, N, K, "f16", "row_col", 0, "pipelined", s2)
            k1_done.wait(60)
            res["t2"] = gp.gemm_stats(sync=True)
        except Exception as e:
            st = gp.gemm_stats(sync=False)
            res["t2_err"] = "%r cuda_error %d at %s" % (e, st["cuda_error"], gp._binding.SITES.get(st["cuda_error_site"]))
        finally:
            t2_read.set()

    th = [threading.Thread(target=t1), threading.Thread(target=t2)]
    for t in th:
        t.start()
    for t in th:
        t.join(120)
    assert "t1_err" not in res and "t2_err" not in res, res
    assert res["t2"]["status"] == 0 and res["t2"]["device_status"] == 0
    assert res["t1"]["status"] == gp.GP_ERR_TIMEOUT and res["t1"]["device_status"] & 0xFF == 1
    check_full("f16", "row_col", A, B, C2.cpu(), K)
    # the next call of thread 1's kind is clean: records are per call, nothing to clear
    gp.gemm_pipelined(tA, tB, C1, M, N, K, "f16", "row_col", 2, "pipelined", s1)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["device_status"] == 0
    check_full("f16", "row_col", A, B, C1.cpu(), K)


def test_release_then_reuse():
    # a stream-K plan uses the workspace; after gemm_release the next call allocates afresh
    M, N, K = 1024, 1024, 4096
    A, B = operands("bf16", "row_col", M, N, K, seed=32)
    tA, tB = to_dev(A, "bf16"), to_dev(B, "bf16")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    gp.gemm_pipelined(tA, tB, C, M, N, K, "bf16", "row_col", 4, "pipelined", stream)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0 and st["plan"]["sk_tiles"] > 0
    first = C.clone()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    gp.release(torch.cuda.current_device())
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after >= free_before + st["plan"]["workspace_bytes"] - (2 << 20)
    C.fill_(0)
    gp.gemm_pipelined(tA, tB, C, M, N, K, "bf16", "row_col", 4, "pipelined", stream)
    assert gp.gemm_stats(sync=True)["status"] == 0
    assert torch.equal(C, first)
    check_full("bf16", "row_col", A, B, C.cpu(), K)
    assert gp.lib().gemm_release(-1) == gp.GP_ERR_ARG


def test_more_streams_than_tracked_workspaces():
    # 72 streams each running a split-K-loop plan (each needs a workspace): the library tracks 64
    # and takes over the least recently used one for the rest; every result is identical
    M, N, K = 1024, 1024, 4096
    A, B = operands("f16", "row_col", M, N, K, seed=33)
    tA, tB = to_dev(A, "f16"), to_dev(B, "f16")
    streams = [torch.cuda.Stream() for _ in range(72)]
    outs = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in streams]
    for s, C in zip(streams, outs):
        gp.gemm_pipelined(tA, tB, C, M, N, K, "f16", "row_col", 4, "pipelined", s)
        st = gp.gemm_stats(sync=False)
        assert st["status"] == 0 and st["plan"]["sk_tiles"] > 0
    for s in streams:
        s.synchronize()
    check_full("f16", "row_col", A, B, outs[0].cpu(), K)
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
    gp.release(torch.cuda.current_device())
