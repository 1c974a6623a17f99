"""Software-pipelined tiled GEMM K-loop for NVIDIA GB300 (sm_103a).

The product is the C-ABI library ``libgemmpipe.so`` (header
``include/gemm_pipelined.h``); this package holds its sources (``csrc/``), the
in-tree build (``build.py``), a thin ctypes binding (``_binding``) with the same
entry-point names, and a torch convenience wrapper ``gemm`` that only
allocates the output and passes pointers.  ``synth`` generates the seeded
synthetic operands.
"""
from ._binding import (  # noqa: F401
    DTYPES, LAYOUTS, VARIANTS, GP_OK, GP_ERR_ARG, GP_ERR_UNSUPPORTED, GP_ERR_SMEM, GP_ERR_CUDA, GP_ERR_TIMEOUT,
    GP_ERR_SIZE, GP_ERR_SCRATCH, GemmError, abi_version, gemm_pipelined, gemm_pipelined_noalloc, gemm_plan,
    gemm_plan_rc, gemm_stats, probe_hbm, probe_peak, release, strerror, lib,
)

_OUT_DTYPE = {"i8": "int32", "f16": "float16", "bf16": "bfloat16", "f32": "float32"}


def gemm(A, B, dtype, layout=None, variant="pipelined", stages=0, out=None, stream=None, **kw):
    """C = A x B for device tensors in storage layout (A: M x K; B: N x K for
    "row_col", K x N for "row_row").  Allocates C with torch if ``out`` is None."""
    import torch
    if layout is None:
        layout = "row_row" if dtype == "f32" else "row_col"
    M, K = A.shape
    N = B.shape[0] if layout == "row_col" else B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=getattr(torch, _OUT_DTYPE[dtype]), device=A.device)
    if stream is None:
        stream = torch.cuda.current_stream(A.device)
    gemm_pipelined(A, B, out, M, N, K, dtype, layout, stages, variant, stream, **kw)
    return out
