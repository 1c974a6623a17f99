#!/usr/bin/env python
"""Benchmark of the software-pipelined tiled GEMM library on GB300.

One step = one GEMM over the workload (all steps of the K-loop hot path:
tile decomposition, prologue, steady-state ring, drain, output epilogue).
Default workload: FP16 GEMM M=N=K=4096, A row-major, B column-major, FP32
accumulate, FP16 out, TMA-ring tcgen05 kernel on CTA pairs at the library's
default depth (6 stages at this shape).  The last line on stdout (rank 0)
is one compact JSON object (under 2 KB): the headline, its roofline, the
end-to-end rate through the C ABI with host buffers, the CPU oracle baseline,
the clocks, and a few scalars of the other configurations (INT8 4096^3 per
call at the library's default, FP32 1024^3, the like-for-like pipelining
gain).  The full sweeps (stage depth per configuration, the BF16
compute/load-ratio sweep with the HBM rows' read/write roof from the
library's own bandwidth probe, the FFMA register-tile sweep) go to a JSON file
(--sweep-out, default bench_sweep.json at the repository root) and, one short line per
configuration, to stdout before the final line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--stages S] [--no-sweep] [--no-sweep-bf16]

--impl reference times the CPU oracle (the reference arm of this build) on a
bounded row sample of the same workload on the host cores.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT8 TOPS and FP16 TFLOPS at 4096^3 (fraction of GB300 dense peak) vs stages"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1920.0, "bf16_tflops_sustained": 1700.0}
ROTATE = 4            # operand/output buffer sets cycled between steps (working set > L2)
L2_BYTES = 129e6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="f16_4096")
    ap.add_argument("--stages", type=int, default=0, help="ring depth (0 = the library's default)")
    ap.add_argument("--variant", default="pipelined")
    ap.add_argument("--one-tile-per-cta", action="store_true",
                    help="run the ring on the register-staged kernels' launch shape (one CTA per tile)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-bf16", action="store_true", default=True,
                    help="include the BF16 stage/ratio sweep (default on)")
    ap.add_argument("--no-sweep-bf16", dest="sweep_bf16", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back steps for the sustained figure (0 = skip)")
    ap.add_argument("--sweep-out", default=os.path.join(ROOT, "bench_sweep.json"),
                    help="file the full sweep results are written to")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["_source"] = "measured (MEASURED_PEAKS.json)"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback (profiling recipe)"
    return d


# ---------------------------------------------------------------------------
# clocks: nvidia-smi sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="gp_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
            os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        import datetime
        def ts(p):
            try:
                return datetime.datetime.strptime(p, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in rows if ts(r[0]) is not None and t0 <= ts(r[0]) <= t1]
        window = "timed"
        if not inside:
            inside, window = rows, "run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        mx = [num(r[3]) for r in inside if num(r[3]) is not None]
        pw = [num(r[4]) for r in inside if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(inside),
                "window": window}


# ---------------------------------------------------------------------------
# device-side timing helpers
# ---------------------------------------------------------------------------
def to_device(torch, x, dtype, dev):
    import numpy as np
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


OUT_TORCH = {"i8": "int32", "f16": "float16", "bf16": "bfloat16", "f32": "float32"}


def device_sets(torch, w, A, B, dev, sets):
    tA = to_device(torch, A, w.dtype, dev)
    tB = to_device(torch, B, w.dtype, dev)
    out = []
    for i in range(sets):
        a = tA if i == 0 else tA.clone()
        b = tB if i == 0 else tB.clone()
        c = torch.empty((w.M, w.N), dtype=getattr(torch, OUT_TORCH[w.dtype]), device=dev)
        out.append((a, b, c))
    return out


def time_kernel(torch, gp, w, bufs, variant, stages, n, stream, **opts):
    """Average device time per launch of n back-to-back launches: CUDA events on `stream` before the
    first and after the last (an event between two launches would stop the next one's set-up from
    overlapping the previous one's tail, as it does in a stream of GEMMs)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        a, b, c = bufs[i % len(bufs)]
        gp.gemm_pipelined(a, b, c, w.M, w.N, w.K, w.dtype, w.layout, stages, variant, stream, **opts)
    e1.record(stream)
    stream.synchronize()
    st = gp.gemm_stats(sync=True)
    if st["status"] != 0:
        raise RuntimeError("kernel status %d" % st["status"])
    ms = e0.elapsed_time(e1) / n
    return ms, ms, st


def isolated_launch_ms(torch, gp, gemm, n, stream):
    """Mean device time of n launches each bracketed by its own pair of CUDA events (no overlap
    with the neighbouring launches)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        evs[i][0].record(stream)
        gemm(i)
        evs[i][1].record(stream)
    stream.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def library_same_shape(torch, w, bufs, stream, n):
    """The vendor library on the same shape, buffers and back-to-back timing, for context only
    (it is not on the product path): torch.matmul (cuBLAS; FP32 with TF32 off) for FP16/BF16/FP32,
    torch._int_mm (cuBLASLt, INT8 -> INT32) for INT8.  Returns (ms per call, how) or (None, why)."""
    def call(i):
        a, b, c = bufs[i % len(bufs)]
        a2 = a.view(w.M, w.K)
        c2 = c.view(w.M, w.N)
        if w.dtype == "i8":
            torch._int_mm(a2, b.view(w.N, w.K).t(), out=c2)
        elif w.layout == "row_col":
            torch.matmul(a2, b.view(w.N, w.K).t(), out=c2)
        else:
            torch.matmul(a2, b.view(w.K, w.N), out=c2)
    how = "torch._int_mm (cuBLASLt)" if w.dtype == "i8" else "torch.matmul (cuBLAS%s)" % (
        ", TF32 off" if w.dtype == "f32" else "")
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        with torch.cuda.stream(stream):
            for i in range(3):
                call(i)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            e0.record(stream)
            for i in range(n):
                call(i)
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) / n, how
    except (RuntimeError, TypeError, AttributeError) as e:
        return None, "%s unavailable: %s" % (how, str(e).splitlines()[0][:160])
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32


def max_over_ranks(torch, dist, x, device):
    """The largest x over all ranks (the slowest rank's time); x itself on one process."""
    if dist is None:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ops_per_step, world, steps, total_ms):
    """Whole-job rate in 1e12 units: every rank runs `steps` independent GEMMs in `total_ms`."""
    return ops_per_step * world * steps / (total_ms * 1e-3) / 1e12


FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12    # SMs x FP32 lanes x FMA x max SM clock
# A timed loop at least this long settles at the power-capped clock and is held to the sustained
# peak.  Sweep rows start rested (see cool()), and a row's loop of tens of milliseconds runs
# mostly above that clock: BF16 8192^2 x 16384, 50 launches of 1.2 ms, measured 1810 TFLOP/s,
# above the 1716 sustained figure and below the 1920 burst one.
SUSTAINED_MS = 1000.0


def compute_peak(kernel, peaks, imma_peak):
    """Peak FLOP/s (or OP/s) of the engine a kernel runs on, in units of 1e12."""
    if kernel.startswith("umma"):
        return peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    if kernel.startswith("imma"):
        return imma_peak
    return FFMA_PEAK_TFLOPS


def roofline_row(w, kernel, ms, peaks, imma_peak):
    """Which roof bounds this GEMM (compute or HBM, whichever takes longer) and the fraction of it reached."""
    t_compute = w.ops / (compute_peak(kernel, peaks, imma_peak) * 1e12)
    t_hbm = w.algorithmic_bytes / (peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]) * 1e9)
    bound = "hbm" if t_hbm > t_compute else ("alu" if kernel.startswith("ffma") else "tensor")
    return bound, round(max(t_compute, t_hbm) / (ms * 1e-3), 4)


def rw_roof_us(w, rw):
    """Least time to move A + B in and C out given the measured copy, pure-read and pure-write
    bandwidths (GB/s): the slowest of the three bounds."""
    return max(w.algorithmic_bytes / rw["copy_gbs"], w.read_bytes / rw["read_gbs"],
               w.write_bytes / rw["write_gbs"]) / 1e3


def hbm_probe(torch, gp, dev, stream, nbytes=2 << 30):
    """Pure-write, pure-read and copy bandwidth of this GPU (GB/s) from the library's own probe
    kernels (16-byte accesses, grid-stride, best over launch shapes; see gemm_probe.h)."""
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    buf.fill_(1)
    torch.cuda.synchronize()
    out = {k + "_gbs": round(gp.probe_hbm(k, buf, stream) / 1e9, 1) for k in ("write", "read", "copy")}
    out["how"] = "gemm_probe_hbm over %d GiB (copy: half onto half), best of 2/4/8 blocks x 512 threads per SM" % (
        nbytes >> 30)
    del buf
    torch.cuda.empty_cache()
    return out


# Pause before each sweep row, so that every row starts at the clocks of a rested GPU: back to
# back, the power draw of the rows before throttles the clock, and whichever depth is measured
# later looks slower (FP16 4096^3, one sequence S = 2..6 then 6, 5, 6, 5: 80.8 us at the first
# S = 5 and 92.5 us at the second).
COOL_S = 0.5


def cool(torch):
    torch.cuda.synchronize()
    time.sleep(COOL_S)


def sweep(torch, gp, dev, stream, names, steps, peaks, imma_peak, rw=None):
    from software_pipelined_tiled_pipeline_gb300 import synth
    from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS
    out = {}
    for name in names:
        w = WORKLOADS[name]
        A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
        bufs = device_sets(torch, w, A, B, dev, ROTATE if w.M * w.K < (1 << 27) else 2)
        unit = "TOPS" if w.dtype == "i8" else "TFLOPS"
        rows = []
        cases = [("nopipe", 1, {}), ("pingpong", 2, {})] + [("pipelined", S, {}) for S in w.stages]
        if w.dtype in ("f16", "bf16"):
            # the same ring on one CTA per 128-row tile, whole tiles only (no pairs, no stream-K)
            cases += [("pipelined", S, {"no_cta_pair": True, "no_stream_k": True}) for S in (4, 6)]
            if w.name == "f16_4096":
                # like for like: the ring on the ping-pong kernel's launch shape (one CTA per
                # 128 x 256 tile, grid = tiles, same smem layout, MMA sequence and epilogue)
                cases += [("pipelined", S, {"one_tile_per_cta": True}) for S in (1, 2, 3, 4)]
            # the caller's promise that the inputs are in place: each launch's loads and MMAs
            # start while the previous launch finishes (only its stores wait)
            cases += [("pipelined", 5, {"inputs_ready": True})]
        if w.dtype == "f32":
            # the caller's promise that the inputs are in place: each launch's loads and FMAs
            # start while the previous launch finishes (only its stores wait)
            cases += [("pipelined", 3, {"inputs_ready": True})]
        if w.dtype == "i8":
            # the TMA ring feeding warp-level IMMA (the ping-pong and no-overlap rows use IMMA too)
            cases += [("pipelined", S, {"i8_engine": "imma"}) for S in w.stages]
            # like for like: the IMMA ring on the ping-pong kernel's launch shape (one CTA per tile)
            cases += [("pipelined", S, {"one_tile_per_cta": True}) for S in (2, 4)]
            # tcgen05 with the int8 -> FP16 conversion overlapped inside the GEMM kernel (one launch)
            cases += [("pipelined", S, {"i8_engine": "tcgen05_overlap"}) for S in (4, 5)]
            # the two-pass engine with successive calls pipelined (the caller promises the inputs are
            # in place: each call's conversion runs beside the previous call's GEMM)
            cases += [("pipelined", 6, {"inputs_ready": True})]
        for variant, S, opts in cases:
            cool(torch)
            time_kernel(torch, gp, w, bufs, variant, S, 3, stream, **opts)      # warm-up
            avg, best, st = time_kernel(torch, gp, w, bufs, variant, S, steps, stream, **opts)
            p = st["plan"]
            rows.append({"variant": variant, "stages": S, "kernel": p["kernel"], "bm": p["bm"], "bn": p["bn"],
                         "cta_pair": p["cta_pair"], **({"options": opts} if opts else {}),
                         "sk_tiles": p["sk_tiles"], "ms": round(avg, 4), unit: round(w.ops / (avg * 1e-3) / 1e12, 2),
                         "regs": st["regs_per_thread"], "smem": p["smem_bytes"]})
            rows[-1]["bound"], rows[-1]["roofline_frac"] = roofline_row(w, p["kernel"], avg, peaks, imma_peak)
            if p["kernel"].startswith("umma") and rows[-1]["bound"] == "tensor" and avg * steps >= SUSTAINED_MS:
                # a loop this long runs at the power-capped clock: its roof is the sustained peak
                sus = dict(peaks, bf16_tflops=peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
                rows[-1]["roofline_frac"] = roofline_row(w, p["kernel"], avg, sus, imma_peak)[1]
                rows[-1]["roof_peak"] = "sustained"
            if rw and rows[-1]["bound"] == "hbm":
                rows[-1]["rw_roof_frac"] = round(rw_roof_us(w, rw) / (avg * 1e3), 4)
        base = next(r for r in rows if r["variant"] == "pingpong")[unit]
        for r in rows:
            r["vs_pingpong"] = round(r[unit] / base, 3) if base else None
            if r.get("options", {}).get("one_tile_per_cta"):
                r["like_for_like"] = True   # same tile, grid and occupancy as the ping-pong row
        out[name] = {"unit": unit, "rows": rows}
        del bufs
        torch.cuda.empty_cache()
    return out


def ffma_tile_sweep(torch, gp, dev, stream, steps=10):
    """The register-tile sweep: FP32 4096^3 on the FFMA ring (S = 3) with each thread tile TM x TN."""
    from software_pipelined_tiled_pipeline_gb300 import synth
    from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS
    w = WORKLOADS["f32_4096"]
    A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    bufs = device_sets(torch, w, A, B, dev, 2)
    rows = []
    for tile in ((4, 8), (8, 4), (8, 8), (8, 16), (16, 8), (16, 16)):
        cool(torch)
        time_kernel(torch, gp, w, bufs, "pipelined", 3, 2, stream, ffma_tile=tile)
        ms, _, st = time_kernel(torch, gp, w, bufs, "pipelined", 3, steps, stream, ffma_tile=tile)
        tf = w.ops / (ms * 1e-3) / 1e12
        rows.append({"tile": "%dx%d" % tile, "threads": st["plan"]["threads"], "ms": round(ms, 4),
                     "TFLOPS": round(tf, 2), "frac_alu": round(tf / FFMA_PEAK_TFLOPS, 4),
                     "regs": st["regs_per_thread"], "spill_bytes": st["local_bytes"]})
    del bufs
    torch.cuda.empty_cache()
    return {"workload": "f32_4096", "stages": 3, "rows": rows}


def int8_default(torch, gp, dev, stream, steps):
    """INT8 4096^3 through the library's default call (stages = 0: the planner's engine and depth),
    back to back on rotating buffers; every call is a full GEMM (its conversion pass included)."""
    from software_pipelined_tiled_pipeline_gb300 import synth
    from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS
    w = WORKLOADS["i8_4096"]
    A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    bufs = device_sets(torch, w, A, B, dev, ROTATE)
    cool(torch)
    time_kernel(torch, gp, w, bufs, "pipelined", 0, 5, stream)
    ms, _, st = time_kernel(torch, gp, w, bufs, "pipelined", 0, steps, stream)
    del bufs
    torch.cuda.empty_cache()
    return {"workload": w.name, "ms": round(ms, 5), "TOPS": round(w.ops / (ms * 1e-3) / 1e12, 2),
            "stages": st["plan"]["stages"], "kernel": st["plan"]["kernel"], "steps": steps}


def compact_line(line, limit=2000):
    """Drop optional keys (last added first) until the JSON line is under `limit` bytes: the
    driver keeps only the tail of stdout."""
    required = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "cpu_baseline", "impl"}
    for key in reversed(list(line)):
        if len(json.dumps(line)) < limit:
            break
        if key not in required:
            del line[key]
    return line


def _code_only(text):
    """Source text without comments and with whitespace collapsed: edits to comments do not
    make a recorded capture stale, edits to code do."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_sha(name):
    """Hash of the code of a kernel source file, the device headers it includes and the planner
    (which sets the schedule, and so the traffic, of every launch)."""
    csrc = os.path.join(ROOT, "software_pipelined_tiled_pipeline_gb300", "csrc")
    h = hashlib.sha256()
    for p in (name, "gp_device.cuh", "gp_internal.h", "api.cu"):
        with open(os.path.join(csrc, p)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel_key, src):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel_key)
    if not d or d.get("source_sha") != source_sha(src):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(w, A, B, seconds):
    """Time the oracle on the first R rows of C, R sized to take about `seconds`."""
    import numpy as np
    import oracle
    run = (lambda rows: oracle.gemm_i8(A, B, w.layout, rows=rows)) if w.dtype == "i8" else \
        (lambda rows: oracle.gemm_ref(A, B, w.dtype, w.layout, rows=rows))
    r = min(16, w.M)
    t0 = time.perf_counter()
    run(np.arange(r))
    t = time.perf_counter() - t0
    R = int(min(w.M, max(r, r * seconds / max(t, 1e-6))))
    t0 = time.perf_counter()
    run(np.arange(R))
    t = time.perf_counter() - t0
    ops = 2.0 * R * w.N * w.K
    return ops / t / 1e12, R, t, oracle.threads()


def run_reference(args, rank):
    from software_pipelined_tiled_pipeline_gb300 import synth
    from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    import numpy as np
    import oracle
    unit = "TOPS" if w.dtype == "i8" else "TFLOPS"
    run = (lambda rows: oracle.gemm_i8(A, B, w.layout, rows=rows)) if w.dtype == "i8" else \
        (lambda rows: oracle.gemm_ref(A, B, w.dtype, w.layout, rows=rows))
    # size one step so the whole --warmup + --steps run takes about 60 s
    budget = 60.0 / max(1, args.steps + args.warmup)
    r = min(8, w.M)
    t0 = time.perf_counter()
    run(np.arange(r))
    t = time.perf_counter() - t0
    R = int(min(w.M, max(1, r * budget / max(t, 1e-6))))
    rows = np.arange(R)
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    el = time.perf_counter() - t0
    value = 2.0 * R * w.N * w.K * args.steps / el / 1e12
    sample = "first %d of %d rows of C per step (%d x %d x %d MACs)" % (R, w.M, R, w.N, w.K)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "M": w.M, "N": w.N, "K": w.K,
                   "sample_rows": R},
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def main():
    args = parse()
    rank, world, local = dist_info()
    if args.impl == "reference":
        return run_reference(args, rank)

    import numpy as np
    import torch
    import software_pipelined_tiled_pipeline_gb300 as gp
    from software_pipelined_tiled_pipeline_gb300 import synth
    from software_pipelined_tiled_pipeline_gb300.workloads import BASE_SEED, WORKLOADS

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    gp.lib()   # fails loudly if the CUDA library is missing

    w = WORKLOADS[args.workload]
    unit = "TOPS" if w.dtype == "i8" else "TFLOPS"
    A, B = synth.operands(w.dtype, w.layout, w.M, w.N, w.K, BASE_SEED)
    bufs = device_sets(torch, w, A, B, dev, ROTATE)
    stream = torch.cuda.Stream(dev)
    peaks = load_peaks()

    def barrier():
        if pg is not None:
            pg.barrier()

    launch_opts = {"one_tile_per_cta": True} if args.one_tile_per_cta else {}

    def gemm(i):
        a, b, c = bufs[i % len(bufs)]
        gp.gemm_pipelined(a, b, c, w.M, w.N, w.K, w.dtype, w.layout, args.stages, args.variant, stream, **launch_opts)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            gemm(i)
        stream.synchronize()
        st = gp.gemm_stats(sync=True)
        if st["status"] != 0:
            raise RuntimeError("warm-up failed: status %d" % st["status"])

        sampler = ClockSampler(local)
        sampler.start()
        # ---- timed region: K steps back to back, barrier + synchronize on both sides ----
        # (events only at its ends: one between launches would stop each launch's set-up
        # from overlapping the previous one's tail)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        wall0 = time.time()
        t_start.record(stream)
        for i in range(args.steps):
            gemm(i)
        t_end.record(stream)
        torch.cuda.synchronize()
        wall1 = time.time()
        barrier()
        clock_rows = sampler.stop()
        st = gp.gemm_stats(sync=True)
        if st["status"] != 0:
            raise RuntimeError("timed region failed: status %d" % st["status"])
        total_ms = t_start.elapsed_time(t_end)
        iso_ms = isolated_launch_ms(torch, gp, gemm, min(args.steps, 50), stream)
    cool(torch)   # the vendor library gets the same rested start as our timed loop
    lib_ms, lib_how = library_same_shape(torch, w, bufs, stream, max(10, min(args.steps, 50)))

    total_ms = max_over_ranks(torch, pg, total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(w.ops, world, args.steps, total_ms)
    kavg = total_ms / args.steps    # average launch duration over the timed region (slowest rank)
    achieved = w.ops / (kavg * 1e-3) / 1e12

    # ---- sustained: the same step back to back for a few seconds (clocks settle under the power cap) ----
    sustained = None
    if args.sustained_s > 0:
        n_s = max(1, int(args.sustained_s * 1e3 / max(kavg, 1e-3)))
        s_sampler = ClockSampler(local)
        s_sampler.start()
        with torch.cuda.stream(stream):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            sw0 = time.time()
            s0.record(stream)
            for i in range(n_s):
                gemm(i)
            s1.record(stream)
            torch.cuda.synchronize()
            sw1 = time.time()
        s_rows = s_sampler.stop()
        st_s = gp.gemm_stats(sync=True)
        if st_s["status"] != 0:
            raise RuntimeError("sustained loop failed: status %d" % st_s["status"])
        s_ms = s0.elapsed_time(s1)
        s_value = w.ops * n_s / (s_ms * 1e-3) / 1e12
        sustained = {"seconds": round(s_ms / 1e3, 2), "launches": n_s, "value": round(s_value, 2), "unit": unit,
                     "clocks": ClockSampler.summarize(s_rows, sw0, sw1)}
        if w.dtype in ("f16", "bf16"):
            sp = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
            sustained.update({"peak": sp, "frac": round(s_value / sp, 4),
                              "peak_source": peaks["_source"] + ": dense bf16 sustained"})

    # ---- end to end: pinned host operands in, result out, every step ----
    # Two device buffer sets and three streams: the inputs of step i+1 are copied in and the
    # result of step i-1 is copied out while step i's GEMM runs (each step still moves its own
    # A and B host -> device and its C device -> host).
    hA = to_device(torch, A, w.dtype, "cpu").pin_memory()
    hB = to_device(torch, B, w.dtype, "cpu").pin_memory()
    hC = [torch.empty((w.M, w.N), dtype=getattr(torch, OUT_TORCH[w.dtype])).pin_memory() for _ in range(2)]
    e2e_steps = max(1, min(args.steps, 50))
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set s are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the GEMM on set s has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # the result of set s is on the host

    def e2e_run(n):
        for i in range(n):
            s_ = i % 2
            dA, dB, dC = bufs[s_]
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(ev_done[s_])          # the GEMM two steps back has read set s
                dA.copy_(hA, non_blocking=True)
                dB.copy_(hB, non_blocking=True)
                ev_in[s_].record(h2d)
            stream.wait_event(ev_in[s_])
            if i >= 2:
                stream.wait_event(ev_out[s_])            # C of set s from two steps back is out
            gp.gemm_pipelined(dA, dB, dC, w.M, w.N, w.K, w.dtype, w.layout, args.stages, args.variant, stream,
                              **launch_opts)
            ev_done[s_].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[s_])
                hC[s_].copy_(dC, non_blocking=True)
                ev_out[s_].record(d2h)
        stream.wait_event(ev_out[(n - 1) % 2])
        if n > 1:
            stream.wait_event(ev_out[(n - 2) % 2])

    e2e_run(2)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(torch, pg, e2e_ms, dev)
    e2e_value = job_throughput(w.ops, world, e2e_steps, e2e_ms)

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0

    plan = st["plan"]
    kernel_src = {"umma": "k_umma.cu", "imma": "k_imma.cu", "ffma": "k_ffma.cu"}[plan["kernel"].split("_")[0]]
    kernel_key = "%s@%s" % (plan["kernel"], w.name)
    imma_peak = gp.probe_peak("imma_s8", stream) / 1e12 if plan["kernel"].startswith("imma") else None
    bound, _ = roofline_row(w, plan["kernel"], kavg, peaks, imma_peak)
    roofline = {"kernel": plan["kernel"], "kernel_avg_ms": round(kavg, 5), "launch_isolated_ms": round(iso_ms, 5),
                "traffic": traffic_for(kernel_key, kernel_src)}
    if bound == "hbm":
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        gbs = w.algorithmic_bytes / (kavg * 1e-3) / 1e9
        rw = hbm_probe(torch, gp, dev, stream)
        roofline.update({"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "algorithmic_bytes": w.algorithmic_bytes,
                         "peak_source": peaks["_source"] + ": copy",
                         "rw_roof_frac": round(rw_roof_us(w, rw) / (kavg * 1e3), 4)})
    else:
        peak = compute_peak(plan["kernel"], peaks, imma_peak)
        roofline.update({"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2),
                         "unit": "TOPS" if w.dtype == "i8" else "TFLOP/s", "frac": round(achieved / peak, 4)})
        if plan["kernel"].startswith("umma") and w.dtype == "i8":
            roofline["peak_source"] = peaks["_source"] + ": dense 16-bit burst (exact FP16 MMAs, conversion included)"
        elif plan["kernel"].startswith("umma"):
            roofline["peak_source"] = peaks["_source"] + ": dense bf16 burst (FP16 at the same rate)"
        elif plan["kernel"].startswith("imma"):
            roofline["peak_source"] = "measured IMMA mma.sync s8 probe (gemm_probe_peak)"
        else:
            roofline["peak_source"] = "152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz"

    clocks = ClockSampler.summarize(clock_rows, wall0, wall1)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout, "variant": args.variant,
                   "stages": plan["stages"], "kernel": plan["kernel"], "tile": "%dx%dx%d" % (
                       plan["bm"], plan["bn"], plan["bk"]), "grid": plan["grid"],
                   "l2": "inputs and output rotated over %d buffer sets (%.0f MiB > 129 MB L2)" % (
                       ROTATE, ROTATE * (A.nbytes + B.nbytes + w.M * w.N * (4 if w.dtype in ("i8", "f32") else 2))
                       / 2 ** 20),
                   "parallelism": "replicas" if world > 1 else "single",
                   **({"one_tile_per_cta": True} if args.one_tile_per_cta else {})},
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": unit, "h2d_bytes_per_step": int(A.nbytes + B.nbytes),
                "d2h_bytes_per_step": int(hC[0].numel() * hC[0].element_size())},
        "gpu_launches": args.steps * (2 if plan["kernel"] == "umma_i8_pair_ring" else 1),
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons"), "samples": clocks.get("samples")},
    }
    if lib_ms:
        line["library_same_shape"] = {"value": round(w.ops / (lib_ms * 1e-3) / 1e12, 1),
                                      "ours_over_library": round(lib_ms / ms_per_step, 3)}
    if sustained:
        line["sustained"] = {k: sustained.get(k) for k in ("value", "frac", "seconds")}
        line["sustained"]["sm_mhz"] = sustained["clocks"].get("sm_mhz")

    extra_steps = max(10, min(args.steps, 50))
    full = {"headline": {"roofline": roofline, "sustained": sustained, "clocks": clocks,
                         "library_same_shape": {"ms_per_call": lib_ms, "how": lib_how}}}
    if not args.no_sweep:
        names = ["f16_4096", "i8_4096", "f32_1024"]
        if args.sweep_bf16:
            names += ["bf16_8192_k256", "bf16_8192_k1024", "bf16_8192_k4096", "bf16_8192_k16384", "bf16_skinny"]
        del bufs
        torch.cuda.empty_cache()
        imma_peak = gp.probe_peak("imma_s8", stream) / 1e12
        rw = hbm_probe(torch, gp, dev, stream) if args.sweep_bf16 else None
        sw = sweep(torch, gp, dev, stream, names, extra_steps, peaks, imma_peak, rw)
        full["hbm_probe"] = rw
        full["sweep"] = sw
        tpeak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        i8 = sw.get("i8_4096")
        if i8:
            # the INT8 headline: the library's default call (stages = 0), timed on its own
            i8d = int8_default(torch, gp, dev, stream, max(20, extra_steps))
            imma = max((r for r in i8["rows"] if r["kernel"] == "imma_ring"), key=lambda r: r["TOPS"])
            promised = [r for r in i8["rows"] if r.get("options", {}).get("inputs_ready")]
            line["int8_4096"] = {"TOPS": i8d["TOPS"], "frac": round(i8d["TOPS"] / tpeak, 4),
                                 "stages": i8d["stages"], "kernel": i8d["kernel"], "launches_per_call": 2,
                                 "imma_ring_TOPS": imma["TOPS"], "imma_ceiling": round(imma_peak, 1)}
            if promised:
                line["int8_4096_inputs_ready"] = {"TOPS": promised[0]["TOPS"],
                                                  "frac": round(promised[0]["TOPS"] / tpeak, 4),
                                                  "caller_promise": True}
            full["int8_default"] = i8d
        f16 = sw.get("f16_4096")
        if f16:
            rows = {(r["variant"], r["stages"], json.dumps(r.get("options", {}), sort_keys=True)): r
                    for r in f16["rows"]}
            pp = rows[("pingpong", 2, "{}")]
            lfl = rows.get(("pipelined", 2, json.dumps({"one_tile_per_cta": True})))
            best = max((r for r in f16["rows"] if r["variant"] == "pipelined" and not r.get("options")),
                       key=lambda r: r["TFLOPS"])
            line["f16_stages"] = {str(r["stages"]): r["TFLOPS"] for r in f16["rows"]
                                  if r["variant"] == "pipelined" and not r.get("options")}
            line["f16_stages"]["pingpong"] = pp["TFLOPS"]
            line["f16_best_stage"] = best["stages"]
            if lfl:
                # the pages' comparison: same tile, grid and occupancy, only the data path differs
                line["pipelining_gain_like_for_like"] = {"f16_ring_s2_over_pingpong": round(
                    lfl["TFLOPS"] / pp["TFLOPS"], 3)}
        f32 = sw.get("f32_1024")
        if f32:
            pf = {r["stages"]: r for r in f32["rows"] if r["variant"] == "pipelined" and not r.get("options")}
            pp32 = next(r for r in f32["rows"] if r["variant"] == "pingpong")
            line["fp32_1024"] = {"TFLOPS": pf[2]["TFLOPS"] if 2 in pf else None,
                                 "frac_alu": pf[2]["roofline_frac"] if 2 in pf else None,
                                 "s2_over_pingpong": pf[2]["vs_pingpong"] if 2 in pf else None,
                                 "pingpong_TFLOPS": pp32["TFLOPS"]}
        full["ffma_peak_probe_tflops"] = round(gp.probe_peak("ffma_f32", stream) / 1e12, 2)
        full["ffma_thread_tile_sweep"] = ffma_tile_sweep(torch, gp, dev, stream)
        for name, d in sw.items():
            short = {"sweep": name, "unit": d["unit"],
                     "rows": [[r["variant"][:4], r["stages"], r[d["unit"]], r["roofline_frac"]] +
                              ([r["options"]] if r.get("options") else []) for r in d["rows"]]}
            print(json.dumps(short), flush=True)

    if not args.no_cpu_baseline and world == 1:
        v, R, t, cores = oracle_sample(w, A, B, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle",
                                "sample": "first %d of %d rows of C in %.1f s" % (R, w.M, t)}
    if args.sweep_out:
        try:
            os.makedirs(os.path.dirname(os.path.abspath(args.sweep_out)), exist_ok=True)
            with open(args.sweep_out, "w") as f:
                json.dump(dict(full, line=line), f, indent=1)
            line["sweep_file"] = os.path.relpath(os.path.abspath(args.sweep_out), ROOT)
        except OSError as e:
            line["sweep_file"] = "not written: %s" % e
    line = compact_line(line)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
