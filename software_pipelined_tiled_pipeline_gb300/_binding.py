"""ctypes binding of the C ABI in include/gemm_pipelined.h.

Argument marshalling only: every step of the GEMM runs in the CUDA kernels of
libgemmpipe.so.  If the library is missing the first call raises -- there is
no fallback of any kind.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgemmpipe.so")

# gp_dtype
GP_I8_I32 = 0
GP_F16_F32ACC_F16OUT = 1
GP_BF16_F32ACC_BF16OUT = 2
GP_F32 = 3
# gp_layout
GP_A_ROW_B_COL = 0
GP_A_ROW_B_ROW = 1
# gp_variant
GP_PINGPONG = 0
GP_PIPELINED = 1
GP_NOPIPE = 2
# error codes
GP_OK = 0
GP_ERR_ARG = -1
GP_ERR_UNSUPPORTED = -2
GP_ERR_SMEM = -3
GP_ERR_CUDA = -4
GP_ERR_TIMEOUT = -5
GP_ERR_SIZE = -6
GP_ERR_SCRATCH = -7
# gp_stats.cuda_error_site
SITES = {1: "device", 2: "event", 3: "capacity", 4: "workspace", 5: "tensor_map", 6: "smem_attr", 7: "launch",
         8: "sync"}

DTYPES = {"i8": GP_I8_I32, "f16": GP_F16_F32ACC_F16OUT, "bf16": GP_BF16_F32ACC_BF16OUT, "f32": GP_F32}
LAYOUTS = {"row_col": GP_A_ROW_B_COL, "row_row": GP_A_ROW_B_ROW}
VARIANTS = {"pingpong": GP_PINGPONG, "pipelined": GP_PIPELINED, "nopipe": GP_NOPIPE}

# exported symbols, in header order
SYMBOLS = ["gemm_pipelined", "gemm_pipelined_ex", "gemm_plan", "gemm_plan_ex", "gemm_stats", "gemm_strerror",
           "gemm_abi_version", "gemm_release", "gemm_pipelined_noalloc", "gemm_probe_peak",
           "gemm_probe_hbm"]


class GpPlan(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32), ("variant", ctypes.c_int32),
        ("stages", ctypes.c_int32), ("bm", ctypes.c_int32), ("bn", ctypes.c_int32), ("bk", ctypes.c_int32),
        ("threads", ctypes.c_int32), ("stage_bytes", ctypes.c_int32), ("ring_bytes", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32), ("persistent", ctypes.c_int32),
        ("grid", ctypes.c_int32), ("tiles", ctypes.c_int64), ("k_tiles", ctypes.c_int64),
        ("compute_load_ratio", ctypes.c_double), ("kernel", ctypes.c_char_p),
        ("dp_tiles", ctypes.c_int32), ("sk_tiles", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("cta_pair", ctypes.c_int32), ("k_splits", ctypes.c_int32), ("half_tiles", ctypes.c_int32),
        ("raster_gm", ctypes.c_int32), ("b_resident", ctypes.c_int32),
    ]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel"] = (self.kernel or b"").decode()
        return d


class GpStats(ctypes.Structure):
    _fields_ = [
        ("plan", GpPlan), ("status", ctypes.c_int32), ("cuda_error", ctypes.c_int32),
        ("regs_per_thread", ctypes.c_int32), ("local_bytes", ctypes.c_int32), ("blocks_per_sm", ctypes.c_int32),
        ("sm_count", ctypes.c_int32), ("device_status", ctypes.c_uint32), ("last_ms", ctypes.c_float),
        ("cuda_error_site", ctypes.c_int32),
    ]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_ if f != "plan"}
        d["plan"] = self.plan.as_dict()
        return d


class GpOptions(ctypes.Structure):
    _fields_ = [
        ("bn", ctypes.c_int32), ("time_kernel", ctypes.c_int32), ("timeout_ns", ctypes.c_uint64),
        ("inject_lost_load", ctypes.c_int32), ("no_stream_k", ctypes.c_int32), ("no_cta_pair", ctypes.c_int32),
        ("i8_engine", ctypes.c_int32), ("ffma_tm", ctypes.c_int32), ("ffma_tn", ctypes.c_int32),
        ("plan_sms", ctypes.c_int32), ("inputs_ready", ctypes.c_int32), ("pair_k_split", ctypes.c_int32),
        ("one_tile_per_cta", ctypes.c_int32), ("raster_gm", ctypes.c_int32),
    ]


_lib = None


class GemmError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, strerror(code), code))


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libgemmpipe.so is not built (run software_pipelined_tiled_pipeline_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    L.gemm_pipelined.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, vp]
    L.gemm_pipelined.restype = ci
    L.gemm_pipelined_ex.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, vp, ctypes.POINTER(GpOptions)]
    L.gemm_pipelined_ex.restype = ci
    L.gemm_plan.argtypes = [i64, i64, i64, ci, ci, ci, ci, ci, ctypes.POINTER(GpPlan)]
    L.gemm_plan.restype = ci
    L.gemm_plan_ex.argtypes = [i64, i64, i64, ci, ci, ci, ci, ctypes.POINTER(GpOptions), ctypes.POINTER(GpPlan)]
    L.gemm_plan_ex.restype = ci
    L.gemm_stats.argtypes = [ctypes.POINTER(GpStats), ci]
    L.gemm_stats.restype = ci
    L.gemm_strerror.argtypes = [ci]
    L.gemm_strerror.restype = ctypes.c_char_p
    L.gemm_abi_version.argtypes = []
    L.gemm_abi_version.restype = ci
    L.gemm_release.argtypes = [ci]
    L.gemm_release.restype = ci
    L.gemm_pipelined_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp]
    L.gemm_pipelined_noalloc.restype = ci
    L.gemm_probe_peak.argtypes = [ci, ctypes.POINTER(ctypes.c_double), vp]
    L.gemm_probe_peak.restype = ci
    L.gemm_probe_hbm.argtypes = [ci, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_double), vp]
    L.gemm_probe_hbm.restype = ci
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()   # torch tensor (device memory)


def _enum(val, table, name):
    if isinstance(val, str):
        if val not in table:
            raise ValueError("unknown %s %r" % (name, val))
        return table[val]
    return int(val)


def release(device=0) -> None:
    """Free the library's device workspaces of `device` (synchronises it)."""
    rc = lib().gemm_release(int(device))
    if rc != GP_OK:
        raise GemmError(rc, "gemm_release")


def strerror(code: int) -> str:
    return lib().gemm_strerror(int(code)).decode()


def abi_version() -> int:
    return lib().gemm_abi_version()


I8_ENGINES = {"default": 0, "imma": 1, "tcgen05_2pass": 2, "tcgen05_overlap": 3}


def _options(bn=0, time_kernel=False, timeout_ns=0, inject_lost_load=False, no_stream_k=False, no_cta_pair=False,
             ffma_tile=None, i8_engine=0, plan_sms=0, inputs_ready=False, pair_k_split=0, one_tile_per_cta=False,
             raster_gm=0):
    opts = GpOptions()
    opts.bn = int(bn)
    opts.time_kernel = 1 if time_kernel else 0
    opts.timeout_ns = int(timeout_ns)
    opts.inject_lost_load = 1 if inject_lost_load else 0
    opts.no_stream_k = 1 if no_stream_k else 0
    opts.no_cta_pair = 1 if no_cta_pair else 0
    opts.i8_engine = _enum(i8_engine, I8_ENGINES, "i8_engine")
    if ffma_tile:
        opts.ffma_tm, opts.ffma_tn = int(ffma_tile[0]), int(ffma_tile[1])
    opts.plan_sms = int(plan_sms)
    opts.inputs_ready = 1 if inputs_ready else 0
    opts.pair_k_split = int(pair_k_split)
    opts.one_tile_per_cta = 1 if one_tile_per_cta else 0
    opts.raster_gm = int(raster_gm)
    return opts


def gemm_pipelined(A, B, C, M, N, K, dtype, layout, stages=0, variant="pipelined", stream=0, *, bn=0,
                   time_kernel=False, timeout_ns=0, inject_lost_load=False, no_stream_k=False, no_cta_pair=False,
                   ffma_tile=None, i8_engine=0, inputs_ready=False, pair_k_split=0, one_tile_per_cta=False,
                   raster_gm=0, check=True) -> int:
    """C = A x B through the C ABI.  A, B, C: device tensors or raw pointers.
    stream: a torch.cuda.Stream, a raw cudaStream_t (int) or 0.
    ffma_tile: (rows, columns) of outputs per thread of the FP32 ring (default 8 x 8).
    i8_engine: INT8 ring engine, a name of I8_ENGINES or its number ("default" lets the planner pick).
    inputs_ready: promise that no work still in flight on the stream writes A or B (see gp_options).
    pair_k_split: 1 = split 256 x 128 tiles' K-loops over two CTA pairs (see gp_options), -1 = never.
    one_tile_per_cta: the ring on the launch shape of the ping-pong kernel (one CTA per tile).
    raster_gm: M blocks per group of the persistent rings' tile raster (0 = the planner's choice)."""
    s = getattr(stream, "cuda_stream", stream)
    opts = _options(bn, time_kernel, timeout_ns, inject_lost_load, no_stream_k, no_cta_pair, ffma_tile, i8_engine,
                    inputs_ready=inputs_ready, pair_k_split=pair_k_split, one_tile_per_cta=one_tile_per_cta,
                    raster_gm=raster_gm)
    rc = lib().gemm_pipelined_ex(_ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), _enum(dtype, DTYPES, "dtype"),
                                 _enum(layout, LAYOUTS, "layout"), int(stages), _enum(variant, VARIANTS, "variant"),
                                 s or None, ctypes.byref(opts))
    if check and rc != GP_OK:
        raise GemmError(rc, "gemm_pipelined")
    return rc


def gemm_pipelined_noalloc(A, B, C, M, N, K, dtype, stages=0, stream=0, check=True) -> int:
    """FP16/BF16 TMA-ring GEMM through the allocation-free entry point: its
    scratch is a fixed device array inside the library (see the C header)."""
    s = getattr(stream, "cuda_stream", stream)
    rc = lib().gemm_pipelined_noalloc(_ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K),
                                      _enum(dtype, DTYPES, "dtype"), int(stages), s or None)
    if check and rc != GP_OK:
        raise GemmError(rc, "gemm_pipelined_noalloc")
    return rc


def gemm_plan(M, N, K, dtype, layout, stages=0, variant="pipelined", bn=0, **opts) -> dict:
    """Tile/stage plan; keyword options as gemm_pipelined (then gemm_plan_ex is used)."""
    p = GpPlan()
    if opts:
        o = _options(bn=bn, **opts)
        rc = lib().gemm_plan_ex(int(M), int(N), int(K), _enum(dtype, DTYPES, "dtype"), _enum(layout, LAYOUTS, "layout"),
                                int(stages), _enum(variant, VARIANTS, "variant"), ctypes.byref(o), ctypes.byref(p))
    else:
        rc = lib().gemm_plan(int(M), int(N), int(K), _enum(dtype, DTYPES, "dtype"), _enum(layout, LAYOUTS, "layout"),
                             int(stages), _enum(variant, VARIANTS, "variant"), int(bn), ctypes.byref(p))
    if rc != GP_OK:
        raise GemmError(rc, "gemm_plan")
    return p.as_dict()


def gemm_plan_rc(M, N, K, dtype, layout, stages=0, variant="pipelined", bn=0) -> int:
    p = GpPlan()
    return lib().gemm_plan(int(M), int(N), int(K), _enum(dtype, DTYPES, "dtype"), _enum(layout, LAYOUTS, "layout"),
                           int(stages), _enum(variant, VARIANTS, "variant"), int(bn), ctypes.byref(p))


def gemm_stats(sync=True) -> dict:
    s = GpStats()
    lib().gemm_stats(ctypes.byref(s), 1 if sync else 0)
    return s.as_dict()


PROBES = {"imma_s8": 0, "ffma_f32": 1}


def probe_peak(kind, stream=0) -> float:
    """Measured ops/s of one instruction path (see include/gemm_probe.h)."""
    out = ctypes.c_double(0.0)
    s = getattr(stream, "cuda_stream", stream)
    rc = lib().gemm_probe_peak(_enum(kind, PROBES, "probe"), ctypes.byref(out), s or None)
    if rc != GP_OK:
        raise GemmError(rc, "gemm_probe_peak")
    return out.value


HBM_PROBES = {"write": 2, "read": 3, "copy": 4}


def probe_hbm(kind, buf, stream=0) -> float:
    """Measured HBM bytes/s of 16-byte stores, loads or a copy over the device tensor `buf`
    (see include/gemm_probe.h; the write and copy probes overwrite it)."""
    out = ctypes.c_double(0.0)
    s = getattr(stream, "cuda_stream", stream)
    rc = lib().gemm_probe_hbm(_enum(kind, HBM_PROBES, "HBM probe"), _ptr(buf), buf.numel() * buf.element_size(),
                              ctypes.byref(out), s or None)
    if rc != GP_OK:
        raise GemmError(rc, "gemm_probe_hbm")
    return out.value
