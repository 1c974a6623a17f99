"""Shared helpers of the GPU parity tests: seeded operands to the device, the
library call through the C ABI into a guarded output buffer, and the
comparison with the CPU oracle (bit-exact for INT8; for floats
max|C - C_ref| <= 1e-2 * sqrt(K/256) * max|C_ref|)."""
import numpy as np
import torch

import oracle
import software_pipelined_tiled_pipeline_gb300 as gp
from software_pipelined_tiled_pipeline_gb300 import synth

OUT_TORCH = {"i8": torch.int32, "f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
GUARD = 4096  # elements of canary on each side of C


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _sentinel(t: torch.Tensor):
    if t.dtype == torch.int32:
        t.fill_(-0x54545455)            # 0xABABABAB
    else:
        t.fill_(float("nan"))


def run(dtype, layout, A, B, M, N, K, variant="pipelined", stages=0, bn=0, **kw):
    """Run the GEMM into the middle of a canary-guarded buffer; return C (host)."""
    tA, tB = to_dev(A, dtype), to_dev(B, dtype)
    buf = torch.empty(M * N + 2 * GUARD, dtype=OUT_TORCH[dtype], device="cuda")
    _sentinel(buf)
    C = buf[GUARD:GUARD + M * N]
    gp.gemm_pipelined(tA, tB, C, M, N, K, dtype, layout, stages, variant, torch.cuda.current_stream(), bn=bn, **kw)
    st = gp.gemm_stats(sync=True)
    assert st["status"] == 0, "status %d (%s), device word %#x, CUDA error %d at %s" % (
        st["status"], gp.strerror(st["status"]), st["device_status"], st["cuda_error"],
        gp._binding.SITES.get(st["cuda_error_site"], st["cuda_error_site"]))
    head, tail = buf[:GUARD].cpu(), buf[GUARD + M * N:].cpu()
    if dtype == "i8":
        assert bool((head == -0x54545455).all()) and bool((tail == -0x54545455).all()), "write outside C"
    else:
        assert bool(torch.isnan(head.float()).all()) and bool(torch.isnan(tail.float()).all()), "write outside C"
    return C.view(M, N).cpu(), st


def host_float(C: torch.Tensor) -> np.ndarray:
    return C.float().numpy().astype(np.float64) if C.dtype in (torch.float16, torch.bfloat16) else \
        C.numpy().astype(np.float64)


def check_full(dtype, layout, A, B, C, K):
    """Compare every element with the oracle."""
    if dtype == "i8":
        ref = oracle.gemm_i8(A, B, layout)
        got = C.numpy()
        bad = np.argwhere(got != ref)
        assert bad.size == 0, "INT8 mismatch at %d places, first %s: got %d want %d" % (
            len(bad), tuple(bad[0]), got[tuple(bad[0])], ref[tuple(bad[0])])
        return 0.0
    ref = oracle.gemm_ref(A, B, dtype, layout)
    got = host_float(C)
    assert np.all(np.isfinite(got)), "non-finite output (unwritten element?)"
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    tol = oracle.tolerance(K, ref, dtype)
    assert err <= tol, "max err %g > tol %g" % (err, tol)
    return err


def check_sampled(dtype, layout, A, B, C, K, rows=None, npts=0, seed=0):
    """Compare listed rows and/or random points with the oracle (large problems)."""
    M, N = C.shape
    rng = np.random.default_rng(seed)
    if rows is not None:
        rows = np.asarray(sorted(set(int(r) for r in rows)), dtype=np.int64)
        if dtype == "i8":
            ref = oracle.gemm_i8(A, B, layout, rows=rows)
            assert np.array_equal(C.numpy()[rows], ref), "INT8 row mismatch"
        else:
            ref = oracle.gemm_ref(A, B, dtype, layout, rows=rows)
            got = host_float(C)[rows]
            err = float(np.max(np.abs(got - ref)))
            tol = oracle.tolerance(K, ref, dtype)
            assert err <= tol, "max err %g > tol %g on sampled rows" % (err, tol)
    if npts:
        r = rng.integers(0, M, npts)
        c = rng.integers(0, N, npts)
        if dtype == "i8":
            ref = oracle.points_i8(A, B, r, c, layout)
            assert np.array_equal(C.numpy()[r, c], ref), "INT8 point mismatch"
        else:
            ref = oracle.points_ref(A, B, dtype, r, c, layout)
            got = host_float(C)[r, c]
            err = float(np.max(np.abs(got - ref)))
            tol = oracle.tolerance(K, ref, dtype)
            assert err <= tol, "max err %g > tol %g on sampled points" % (err, tol)


def operands(dtype, layout, M, N, K, seed, dist=None):
    return synth.operands(dtype, layout, M, N, K, seed, dist=dist)
