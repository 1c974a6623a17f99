"""Host-side checks of the C ABI (no GPU): the library loads and exports every
symbol the header declares, argument errors are reported before anything is
launched, and the tile / stage / shared-memory choice follows the budget
rules ("pipeline-gpu-kernel", Step 1 and Step 2)."""
import ctypes
import json
import os
import re

import pytest

from software_pipelined_tiled_pipeline_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def gp():
    gbuild.build()
    import software_pipelined_tiled_pipeline_gb300 as mod
    mod.lib()
    return mod


def header_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(gp):
    names = header_functions()
    assert "gemm_pipelined" in names and "gemm_stats" in names
    L = ctypes.CDLL(gbuild.LIB)
    for n in names:
        assert hasattr(L, n), "symbol %s declared in include/ but not exported" % n
    from software_pipelined_tiled_pipeline_gb300 import _binding
    assert sorted(_binding.SYMBOLS) == sorted(names)


def test_version_and_strerror(gp):
    assert gp.abi_version() == 10700
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert gp.strerror(code) and "unknown" not in gp.strerror(code)
    assert "unknown" in gp.strerror(-99)


def test_struct_sizes_match_c_layout(tmp_path):
    # the ctypes mirrors against the header as a C compiler lays it out (sizes and field offsets)
    import shutil
    import subprocess
    from software_pipelined_tiled_pipeline_gb300 import _binding as b
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    include = os.path.join(ROOT, "include")
    src = tmp_path / "sizes.c"
    checks = [("gp_plan", b.GpPlan), ("gp_stats", b.GpStats), ("gp_options", b.GpOptions)]
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "gemm_pipelined.h"', "int main(void) {"]
    for cname, cls in checks:
        lines.append('  printf("%%s %%zu\\n", "%s", sizeof(%s));' % (cname, cname))
        for f, _ in cls._fields_:
            lines.append('  printf("%%s.%%s %%zu\\n", "%s", "%s", offsetof(%s, %s));' % (cname, f, cname, f))
    lines.append("  return 0;\n}")
    src.write_text("\n".join(lines))
    exe = tmp_path / "sizes"
    subprocess.run([cc, "-I", include, str(src), "-o", str(exe)], check=True)
    out = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                          text=True).stdout.splitlines())
    for cname, cls in checks:
        assert int(out[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(out["%s.%s" % (cname, f)]) == getattr(cls, f).offset, (cname, f)


@pytest.mark.parametrize("args,code", [
    (dict(dtype=7), -1), (dict(layout=5), -1), (dict(variant=9), -1),
    (dict(M=-1), -1), (dict(K=-3), -1), (dict(M=1 << 31), -6),
    (dict(stages=9), -1), (dict(stages=-1), -1),
    (dict(variant=0, stages=3), -1), (dict(variant=2, stages=2), -1),
    (dict(dtype=3, layout=0), -2), (dict(dtype=0, layout=1), -2),
    (dict(bn=96), -2), (dict(bn=256, stages=8), -3), (dict(bn=-1), -1),
])
def test_plan_argument_errors(gp, args, code):
    a = dict(M=256, N=256, K=256, dtype=1, layout=0, stages=4, variant=1, bn=0)
    a.update(args)
    rc = gp.gemm_plan_rc(a["M"], a["N"], a["K"], a["dtype"], a["layout"], a["stages"], a["variant"], a["bn"])
    assert rc == code


def test_call_argument_errors_need_no_device(gp):
    L = gp.lib()
    f = L.gemm_pipelined
    ok_ptr = 0x10000
    # null output with a non-empty result
    assert f(ok_ptr, ok_ptr, None, 64, 64, 64, 1, 0, 4, 1, None) == gp.GP_ERR_ARG
    assert f(None, ok_ptr, ok_ptr, 64, 64, 64, 1, 0, 4, 1, None) == gp.GP_ERR_ARG
    # misaligned base pointer
    assert f(ok_ptr + 8, ok_ptr, ok_ptr, 64, 64, 64, 1, 0, 4, 1, None) == gp.GP_ERR_UNSUPPORTED
    # K not a multiple of 16 bytes of row for INT8 / FP16, N rule for C rows
    assert f(ok_ptr, ok_ptr, ok_ptr, 64, 64, 40, 0, 0, 4, 1, None) == gp.GP_ERR_UNSUPPORTED
    assert f(ok_ptr, ok_ptr, ok_ptr, 64, 64, 36, 1, 0, 4, 1, None) == gp.GP_ERR_UNSUPPORTED
    assert f(ok_ptr, ok_ptr, ok_ptr, 64, 60, 64, 1, 0, 4, 1, None) == gp.GP_ERR_UNSUPPORTED
    assert f(ok_ptr, ok_ptr, ok_ptr, 64, 62, 64, 3, 1, 2, 1, None) == gp.GP_ERR_UNSUPPORTED
    # empty output: nothing to do, no device touched
    assert f(None, None, None, 0, 64, 64, 1, 0, 4, 1, None) == gp.GP_OK
    assert f(None, None, None, 64, 0, 64, 0, 0, 4, 1, None) == gp.GP_OK
    st = gp.gemm_stats(sync=False)
    assert st["status"] == 0


def test_hbm_probe_argument_errors_need_no_device(gp):
    import ctypes
    f = gp.lib().gemm_probe_hbm
    out = ctypes.c_double(0.0)
    ok_ptr, mib = 0x10000, 1 << 20
    assert f(2, None, mib, ctypes.byref(out), None) == gp.GP_ERR_ARG          # no buffer
    assert f(2, ok_ptr, mib, None, None) == gp.GP_ERR_ARG                     # no output
    assert f(5, ok_ptr, mib, ctypes.byref(out), None) == gp.GP_ERR_ARG        # not an HBM probe
    assert f(0, ok_ptr, mib, ctypes.byref(out), None) == gp.GP_ERR_ARG        # (the IMMA probe kind)
    assert f(3, ok_ptr + 8, mib, ctypes.byref(out), None) == gp.GP_ERR_ARG    # misaligned
    assert f(3, ok_ptr, mib - 32, ctypes.byref(out), None) == gp.GP_ERR_ARG   # under 1 MiB
    assert f(4, ok_ptr, mib + 16, ctypes.byref(out), None) == gp.GP_ERR_ARG   # not whole 32-byte pairs
    with pytest.raises(ValueError):
        gp.probe_hbm("sum", None)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6])
def test_umma_pairs_up_to_six_stages(gp, S):
    # CTA pair: 256 x 256 tile per pair, each CTA 128 rows of A and 128 of B = 32 KB per K step
    p = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined")
    assert p["cta_pair"] == 1 and p["kernel"] == "umma_pair_ring"
    assert (p["bm"], p["bn"], p["bk"], p["stages"]) == (256, 256, 64, S)
    assert p["stage_bytes"] == 2 * 128 * 64 * 2 and p["ring_bytes"] == S * p["stage_bytes"]
    assert 232448 // 2 < p["smem_bytes"] <= 232448
    assert p["tmem_cols"] == 512 and p["persistent"] == 1
    assert p["tiles"] == 16 * 16 and p["k_tiles"] == 64
    # per CTA: 2*128*256*64 / ((128 + 128) * 64 * 2) FLOP per byte loaded
    assert p["compute_load_ratio"] == pytest.approx(128.0)


def test_default_depth_follows_k(gp):
    # FP16/BF16 ring: 4 stages at K <= 256 (one CTA per tile), 6 on the 256 x 256 pair tile at every longer K
    for K, S in ((256, 4), (1024, 6), (2048, 6), (4096, 6), (16384, 6)):
        assert gp.gemm_plan(8192, 8192, K, "bf16", "row_col", 0, "pipelined")["stages"] == S, K
    assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 0, "pipelined")["stages"] == 6
    # 64 < N <= 128 on the 256 x 128 pair tile: the deepest ring (with the K split: 5, see below)
    p = gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined", pair_k_split=-1)
    assert (p["stages"], p["cta_pair"], p["bn"]) == (8, 1, 128)


def test_ffma_thread_tiles(gp):
    # the register-tile sweep: outputs per thread TM x TN of the 128 x 128 CTA tile, plus a producer warp
    for (tm, tn) in ((4, 8), (8, 4), (8, 8), (8, 16), (16, 8), (16, 16)):
        p = gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 3, "pipelined", ffma_tile=(tm, tn))
        assert p["threads"] == (128 // tm) * (128 // tn) + 32 and (p["bm"], p["bn"], p["bk"]) == (128, 128, 32)
        assert p["stage_bytes"] == (128 * 32 + 32 * 128) * 4
    # the ring takes 32 K steps per slot up to 6 slots, 16 at 7-8 (eight 32 KB slots would not fit)
    for S, bk in ((1, 32), (6, 32), (7, 16), (8, 16)):
        p = gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", S, "pipelined")
        assert (p["bk"], p["stage_bytes"], p["ring_bytes"]) == (bk, (128 * bk + bk * 128) * 4, S * (128 * bk + bk * 128) * 4)
        assert p["smem_bytes"] <= 232448
    # the register-staged baselines keep 8 K steps per tile (their thread-to-element mapping)
    for v in ("pingpong", "nopipe"):
        q = gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 0, v)
        assert (q["bk"], q["stage_bytes"]) == (8, (128 * 8 + 8 * 128) * 4)
    for bad in ((4, 4), (8, 2), (32, 8), (12, 8)):
        with pytest.raises(gp.GemmError):
            gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 3, "pipelined", ffma_tile=bad)
    # the register-staged variants build the pages' 8 x 8 only
    with pytest.raises(gp.GemmError):
        gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 2, "pingpong", ffma_tile=(16, 8))
    assert gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 2, "pingpong", ffma_tile=(8, 8))["threads"] == 256


def test_short_k_runs_one_cta_per_tile(gp):
    # K <= 256: a few K steps per tile, C's write dominates -- one CTA per 128 x 256 tile at 4 stages
    for K in (64, 200, 256):
        p = gp.gemm_plan(8192, 8192, K, "bf16", "row_col", 0, "pipelined")
        assert (p["cta_pair"], p["bn"], p["stages"]) == (0, 256, 4), K
        # (with SMs queried, K = 200 and 256 keep B in the ring at one slot per K step: still 4)
    p = gp.gemm_plan(8192, 8192, 320, "bf16", "row_col", 0, "pipelined")
    assert (p["cta_pair"], p["stages"]) == (1, 6)
    assert gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 6, "pipelined")["cta_pair"] == 0
    assert gp.gemm_plan(8192, 128, 256, "bf16", "row_col", 0, "pipelined")["stages"] == 6   # N <= 128: BN 128


def test_b_resident_plan(gp):
    # a K-loop of 2-4 steps that fills the ring, whole tiles, more tiles than SMs: one slot per K step,
    # contiguous tile runs in M-block-fastest order, B kept in the ring while the N block repeats
    kw = dict(plan_sms=152)
    for K, kt in ((128, 2), (192, 3), (200, 4), (256, 4)):
        p = gp.gemm_plan(8192, 8192, K, "bf16", "row_col", 0, "pipelined", **kw)
        assert (p["b_resident"], p["stages"], p["k_tiles"], p["raster_gm"], p["bn"], p["cta_pair"]) == \
            (1, kt, kt, 64, 256, 0), K
        assert p["ring_bytes"] == kt * (128 + 256) * 64 * 2
        assert p["smem_bytes"] == max(1024 + p["ring_bytes"] + 32768 + 256, 232448 // 2 + 1024)
    assert gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 4, "pipelined", **kw)["b_resident"] == 1
    assert gp.gemm_plan(2000, 5000, 192, "f16", "row_col", 0, "pipelined", **kw)["b_resident"] == 1
    # streamed: one K step, a depth other than the K-loop, a raster chosen by the caller, one tile per
    # CTA, fewer tiles than SMs, and K beyond the ring (the CTA pair)
    assert gp.gemm_plan(8192, 8192, 64, "bf16", "row_col", 0, "pipelined", **kw)["b_resident"] == 0
    assert gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 3, "pipelined", **kw)["b_resident"] == 0
    assert gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 0, "pipelined", raster_gm=8, **kw)["b_resident"] == 0
    assert gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 0, "pipelined", one_tile_per_cta=True,
                        **kw)["b_resident"] == 0
    assert gp.gemm_plan(1024, 1024, 256, "bf16", "row_col", 0, "pipelined", **kw)["b_resident"] == 0
    assert gp.gemm_plan(8192, 8192, 512, "bf16", "row_col", 0, "pipelined", **kw)["b_resident"] == 0
    assert gp.gemm_plan(4096, 4096, 256, "i8", "row_col", 0, "pipelined", **kw)["b_resident"] == 0


@pytest.mark.parametrize("S", range(1, 9))
def test_umma_single_cta_widths_follow_the_budget(gp, S):
    # one CTA per 128 x BN tile: the widths the 227 KB budget admits at this depth
    for b in (256, 128, 64):
        fits = 1024 + S * (128 + b) * 64 * 2 + 32768 + 256 <= 232448
        rc = gp.gemm_plan_rc(4096, 4096, 4096, "f16", "row_col", S, "pipelined", bn=b)
        if b == 256 and S <= 6:
            assert rc == 0 and gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined", bn=b)["cta_pair"] == 1
            continue
        assert rc == (0 if fits else -3), (S, b, rc)
        if fits:
            q = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined", bn=b)
            assert q["cta_pair"] == 0 and q["bm"] == 128 and q["bn"] == b
            assert q["stage_bytes"] == (128 + b) * 64 * 2 and q["tmem_cols"] == 2 * b
            assert q["tiles"] == 32 * (4096 // b)
    if S > 6:
        # the 256 x 256 pair tile does not fit 7-8 stages; the 256 x 128 pair tile does
        p = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined")
        assert p["cta_pair"] == 1 and (p["bm"], p["bn"]) == (256, 128)
        assert p["stage_bytes"] == (128 + 64) * 64 * 2 and p["tmem_cols"] == 256
        assert p["smem_bytes"] <= 232448 and p["tiles"] == 16 * 32


def test_pair_tile_128_for_narrow_n(gp):
    # 64 < N <= 128: 256 x 128 tile per CTA pair (each CTA 128 rows of A, 64 rows of B), up to 8 stages
    for S in range(1, 9):
        p = gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", S, "pipelined")
        assert p["kernel"] == "umma_pair_ring" and (p["bm"], p["bn"], p["stages"]) == (256, 128, S)
        assert p["ring_bytes"] == S * 24576
    # N <= 64, M <= 128, K <= 256 or an explicit width: one CTA per tile
    assert gp.gemm_plan(8192, 64, 8192, "bf16", "row_col", 6, "pipelined")["cta_pair"] == 0
    assert gp.gemm_plan(128, 128, 8192, "bf16", "row_col", 6, "pipelined")["cta_pair"] == 0
    assert gp.gemm_plan(8192, 128, 256, "bf16", "row_col", 6, "pipelined")["cta_pair"] == 0
    assert gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 6, "pipelined", bn=128)["cta_pair"] == 0


@pytest.mark.parametrize("S,bn", [(1, 128), (4, 128), (6, 128), (7, 128), (8, 64)])
def test_imma_tile_shrinks_with_stages(gp, S, bn):
    p = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined", i8_engine="imma")
    assert p["kernel"] == "imma_ring" and p["cta_pair"] == 0
    assert p["bn"] == bn and p["bk"] == 128 and p["stage_bytes"] == (128 + bn) * 128
    assert p["k_tiles"] == 32 and p["smem_bytes"] <= 232448


@pytest.mark.parametrize("S", range(1, 7))
def test_int8_on_tcgen05_plan(gp, S):
    # default INT8 ring: FP16 operands on CTA pairs, 256 x 256 tile, 32 KB per CTA per K step of 64
    p = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined")
    assert p["kernel"] == "umma_i8_pair_ring" and p["cta_pair"] == 1
    assert (p["bm"], p["bn"], p["bk"], p["stages"]) == (256, 256, 64, S)
    assert p["stage_bytes"] == (128 + 128) * 64 * 2 and p["tmem_cols"] == 512 and p["threads"] == 320
    assert p["smem_bytes"] <= 232448 and p["k_tiles"] == 64 and p["tiles"] == 16 * 16
    # FP16 copies of A and B, after the stream-K partial tiles (two 128 x 256 int32 slots per CTA) if any
    partials = p["grid"] * 2 * 128 * 256 * 4 if p["sk_tiles"] > 0 else 0
    assert p["workspace_bytes"] == (4096 + 4096) * 4096 * 2 + partials
    # bn=64 or an IMMA request selects the warp-level IMMA ring
    assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined", bn=64)["kernel"] == "imma_ring"
    for deep in (7, 8):   # rings deeper than the pair tile allows run on IMMA
        assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", deep, "pipelined")["kernel"] == "imma_ring"
    assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined", bn=128)["kernel"] == "imma_ring"


@pytest.mark.parametrize("S", range(1, 7))
def test_int8_overlap_engine_plan(gp, S):
    # the two-pass engine's ring, tile and FP16 copies, in one 512-thread kernel that writes
    # the copies itself through an int8 staging ring of 8 KB slots (as many as fit, up to 8,
    # at least 2), with whole tiles only
    p = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined", i8_engine="tcgen05_overlap")
    q = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", S, "pipelined", i8_engine="tcgen05_2pass")
    assert q["kernel"] == "umma_i8_pair_ring" and q["threads"] == 320
    if S == 6:   # no room left for staging: the two-pass engine runs
        assert p == q
        return
    assert p["kernel"] == "umma_i8_overlap_pair_ring" and p["threads"] == 512 and p["sk_tiles"] == 0
    for key in ("bm", "bn", "bk", "stages", "stage_bytes", "ring_bytes", "tmem_cols", "tiles", "grid", "cta_pair",
                "compute_load_ratio", "workspace_bytes"):
        assert p[key] == q[key], key
    fixed = 1024 + 32768 + 256 + 384   # alignment slack, epilogue staging, ring and hand-off barriers
    slots = min(8, (232448 - fixed - S * 32768) // 8192)
    assert slots >= 2 and p["smem_bytes"] == max(fixed + S * 32768 + slots * 8192, 232448 // 2 + 1024) <= 232448
    assert p["workspace_bytes"] == (4096 + 4096) * 4096 * 2
    small = gp.gemm_plan(256, 256, 1024, "i8", "row_col", S, "pipelined", i8_engine="tcgen05_overlap")
    assert small["sk_tiles"] == 0 and small["dp_tiles"] == 1
    assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 7, "pipelined",
                        i8_engine="tcgen05_overlap")["kernel"] == "imma_ring"


def test_int8_overlap_default_depth(gp):
    p = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 0, "pipelined", i8_engine="tcgen05_overlap")
    assert p["kernel"] == "umma_i8_overlap_pair_ring" and p["stages"] == 5


def test_small_n_picks_narrow_tile(gp):
    assert gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 4, "pipelined")["bn"] == 128
    assert gp.gemm_plan(8192, 64, 8192, "bf16", "row_col", 4, "pipelined")["bn"] == 64
    assert gp.gemm_plan(256, 100 + 4, 256, "i8", "row_col", 4, "pipelined", i8_engine="imma")["bn"] == 128


def test_default_stages_and_variant_stage_rules(gp):
    assert gp.gemm_plan(512, 512, 512, "f16", "row_col", 0, "pipelined")["stages"] == 6
    assert gp.gemm_plan(512, 512, 512, "i8", "row_col", 0, "pipelined")["stages"] == 6
    assert gp.gemm_plan(512, 512, 512, "i8", "row_col", 0, "pipelined", i8_engine="imma")["stages"] == 4
    assert gp.gemm_plan(512, 512, 512, "f16", "row_col", 0, "pingpong")["stages"] == 2
    assert gp.gemm_plan(512, 512, 512, "f16", "row_col", 0, "nopipe")["stages"] == 1
    assert gp.gemm_plan(512, 512, 512, "f32", "row_row", 0, "pipelined")["stages"] == 3


def test_compute_load_ratio_is_the_published_formula(gp):
    for dtype, layout, esize, bn in (("f16", "row_col", 2, 128), ("i8", "row_col", 1, 64), ("f32", "row_row", 4, 0)):
        p = gp.gemm_plan(4096, 4096, 4096, dtype, layout, 2, "pipelined", bn=bn)
        bm, bn, bk = p["bm"], p["bn"], p["bk"]
        assert p["compute_load_ratio"] == pytest.approx(2 * bm * bn * bk / ((bm * bk + bk * bn) * esize))
    # FP16 128x64x64 on one CTA: 2*128*64*64 / ((128*64 + 64*64) * 2) FLOP per byte
    p = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 7, "pipelined", bn=64)
    assert p["compute_load_ratio"] == pytest.approx(2 * 128 * 64 * 64 / ((128 * 64 + 64 * 64) * 2))
    p = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 4, "pipelined", bn=128)
    assert p["compute_load_ratio"] == pytest.approx(64.0)


def test_ffma_tile_matches_published_kernel_table(gp):
    g = json.load(open(os.path.join(GOLDEN, "p1_kernel_table.json")))
    t = g["tile"]
    M = g["problem"]["M"]
    nop = gp.gemm_plan(M, M, M, "f32", "row_row", 1, "nopipe")
    pp = gp.gemm_plan(M, M, M, "f32", "row_row", 2, "pingpong")
    ring2 = gp.gemm_plan(M, M, M, "f32", "row_row", 2, "pipelined")
    assert (nop["bm"], nop["bn"], nop["bk"], nop["threads"]) == (t["bm"], t["bn"], t["bk"], t["threads"])
    assert nop["k_tiles"] == g["k_tiles"]
    kb = g["static_smem_per_block_kb"]
    assert round(nop["ring_bytes"] / 1000, 2) == kb["baseline"]
    assert round(pp["ring_bytes"] / 1000, 2) == kb["ping_pong"]
    # the TMA ring takes 32 K steps per slot where the pages' kernels take 8: per 8 K steps its two
    # slots hold what the pages' two-stage buffer holds
    assert ring2["bk"] == 4 * t["bk"]
    assert round(ring2["ring_bytes"] * t["bk"] / ring2["bk"] / 1000, 2) == kb["cp_async_2stage"]


def test_throughput_formula_matches_published_benchmark():
    from software_pipelined_tiled_pipeline_gb300.workloads import Workload
    g = json.load(open(os.path.join(GOLDEN, "p1_kernel_table.json")))
    M = g["problem"]["M"]
    w = Workload("p1", "f32", "row_row", M, M, M)
    for row in g["benchmark"]:
        gflops = w.ops / (row["avg_ms"] * 1e-3) / 1e9
        # the printed time has 3 decimals: +-0.0005 ms
        slack = w.ops / ((row["avg_ms"] - 0.0005) * 1e-3) / 1e9 - gflops
        assert abs(gflops - row["gflops"]) <= slack + 0.05


def test_double_buffer_rule_matches_published_example():
    g = json.load(open(os.path.join(GOLDEN, "p2_smem_budget.json")))
    # single buffer 2 KB + 2 KB -> doubled 8 KB
    assert 2 * g["single_buffer_kb"] == g["double_buffer_kb"]


def test_no_512_wide_tile(gp):
    # no tile is 512 columns wide: every dtype and layout refuses bn = 512
    for M, N, K, dt, lay in [(4096, 4096, 4096, "f16", "row_col"), (4096, 4096, 4096, "bf16", "row_col"),
                             (4096, 4096, 256, "f16", "row_col"), (4096, 4096, 4096, "f32", "row_row"),
                             (4096, 4096, 4096, "i8", "row_col"), (4096, 128, 4096, "bf16", "row_col")]:
        assert gp.gemm_plan_rc(M, N, K, dt, lay, 0, "pipelined", bn=512) == gp.GP_ERR_UNSUPPORTED


def test_one_tile_per_cta_plan(gp):
    # the ring on the ping-pong kernel's launch shape: one CTA per 128 x 256 tile, grid = tiles,
    # not persistent, no pairs, no stream-K; same tile as the register-staged variants
    for S in (1, 2, 3, 4):
        r = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined", plan_sms=152, one_tile_per_cta=True)
        assert (r["kernel"], r["bm"], r["bn"], r["bk"], r["cta_pair"]) == ("umma_ring", 128, 256, 64, 0)
        assert (r["grid"], r["tiles"], r["persistent"], r["sk_tiles"]) == (512, 512, 0, 0)
    pp = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 2, "pingpong", plan_sms=152)
    assert (pp["bm"], pp["bn"], pp["bk"], pp["grid"]) == (128, 256, 64, 512)
    i = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 4, "pipelined", plan_sms=152, one_tile_per_cta=True)
    ip = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 2, "pingpong", plan_sms=152)
    assert (i["kernel"], i["bm"], i["bn"], i["persistent"]) == ("imma_ring", ip["bm"], ip["bn"], 0)
    assert i["tiles"] == ip["tiles"] == ip["grid"]
    f = gp.gemm_plan(1024, 1024, 1024, "f32", "row_row", 3, "pipelined", plan_sms=152, one_tile_per_cta=True)
    assert (f["k_splits"], f["grid"]) == (1, 64)


def test_raster_group_plan(gp):
    # one raster group over all row blocks while their A panels fit the L2 budget, else groups of 8
    kw = dict(plan_sms=152)
    assert gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined", **kw)["raster_gm"] == 16
    assert gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 0, "pipelined", **kw)["raster_gm"] == 16
    assert gp.gemm_plan(8192, 8192, 4096, "bf16", "row_col", 0, "pipelined", **kw)["raster_gm"] == 8
    assert gp.gemm_plan(4096, 4096, 16384, "f16", "row_col", 0, "pipelined", **kw)["raster_gm"] == 8
    assert gp.gemm_plan(1000, 1800, 1040, "bf16", "row_col", 0, "pipelined", **kw)["raster_gm"] == 4
    assert gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined", raster_gm=3, **kw)["raster_gm"] == 3
    with pytest.raises(gp.GemmError) as ex:
        gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined", raster_gm=-1)
    assert ex.value.code == gp.GP_ERR_ARG


def test_pair_k_split_plan(gp):
    # pair_k_split = 1: each 256 x 128 tile on a cluster of two CTA pairs, each pair half of the
    # K-loop; no stream-K; at most 5 stages (the 64 KB receive buffer)
    kw = dict(plan_sms=152, pair_k_split=1)
    p = gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined", **kw)
    assert (p["kernel"], p["cta_pair"], p["bm"], p["bn"], p["stages"]) == ("umma_pair_ksplit_ring", 3, 256, 128, 5)
    assert (p["tiles"], p["grid"], p["dp_tiles"], p["sk_tiles"], p["workspace_bytes"]) == (32, 128, 32, 0, 0)
    assert p["smem_bytes"] <= 232448
    # the planner's choice: 32 tiles (more than 152/8, at most 152/4) and 128 K steps -> the K split
    d = gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined", plan_sms=152)
    assert (d["cta_pair"], d["stages"]) == (3, 5)
    assert gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined", plan_sms=152,
                        pair_k_split=-1)["cta_pair"] == 1
    # fewer tiles (stream-K over all pairs), short K-loops, or no device: CTA pairs
    assert gp.gemm_plan(2048, 128, 8192, "bf16", "row_col", 0, "pipelined", plan_sms=152)["cta_pair"] == 1
    assert gp.gemm_plan(8192, 128, 1024, "bf16", "row_col", 0, "pipelined", plan_sms=152)["cta_pair"] == 1
    assert gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined")["cta_pair"] == 1
    with pytest.raises(gp.GemmError):   # 6 stages leave no room for the receive buffer
        gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 6, "pipelined", **kw)
    for M, N, K, dt in [(4096, 4096, 4096, "f16"), (8192, 128, 256, "bf16"), (4096, 128, 4096, "i8")]:
        assert gp.gemm_plan_rc(M, N, K, dt, "row_col", 0, "pipelined") == 0
        with pytest.raises(gp.GemmError):
            gp.gemm_plan(M, N, K, dt, "row_col", 0, "pipelined", pair_k_split=1)
    with pytest.raises(gp.GemmError):
        gp.gemm_plan(8192, 128, 8192, "bf16", "row_col", 0, "pipelined", pair_k_split=2)


def test_planner_for_a_152_sm_gb300(gp):
    # the launch-time decisions, planned for a GB300's 152 SMs (76 CTA pairs) without a device
    kw = dict(plan_sms=152)
    f16 = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined", **kw)
    # 256 tiles on 76 pairs: three whole waves, the 28 tiles left over split evenly (stream-K)
    assert (f16["kernel"], f16["stages"], f16["bn"], f16["grid"]) == ("umma_pair_ring", 6, 256, 152)
    assert (f16["tiles"], f16["dp_tiles"], f16["sk_tiles"]) == (256, 228, 28)
    assert f16["workspace_bytes"] == 152 * 2 * 128 * 256 * 4
    # a ring of at most 4 slots splits the last full wave too: two whole waves, 104 split tiles
    for S in (2, 3, 4):
        q = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", S, "pipelined", **kw)
        assert (q["dp_tiles"], q["sk_tiles"], q["grid"]) == (152, 104, 152), S
    q = gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 5, "pipelined", **kw)
    assert (q["dp_tiles"], q["sk_tiles"]) == (228, 28)
    # 8192^2 x 16384 on the 6-slot ring: 1024 tiles, 13 whole waves, 36 split tiles
    big = gp.gemm_plan(8192, 8192, 16384, "bf16", "row_col", 0, "pipelined", **kw)
    assert (big["tiles"], big["dp_tiles"], big["sk_tiles"]) == (1024, 988, 36)
    i8 = gp.gemm_plan(4096, 4096, 4096, "i8", "row_col", 0, "pipelined", **kw)
    # three whole waves, then the 28 tiles left over as 56 half tiles on 56 pairs
    assert (i8["kernel"], i8["stages"], i8["grid"], i8["sk_tiles"]) == ("umma_i8_pair_ring", 6, 152, 0)
    assert (i8["dp_tiles"], i8["half_tiles"]) == (228, 28)
    assert i8["workspace_bytes"] == (4096 + 4096) * 4096 * 2
    few = gp.gemm_plan(768, 2048, 8192, "i8", "row_col", 0, "pipelined", **kw)
    # 24 tiles do not fill one wave: every K-loop is split over the 76 pairs, exact int32 partials
    assert (few["dp_tiles"], few["sk_tiles"], few["half_tiles"], few["grid"]) == (0, 24, 0, 152)
    assert few["workspace_bytes"] == 152 * 2 * 128 * 256 * 4 + (768 + 2048) * 8192 * 2
    full = gp.gemm_plan(256 * 76, 256, 1024, "i8", "row_col", 0, "pipelined", **kw)
    assert (full["tiles"], full["dp_tiles"], full["sk_tiles"], full["half_tiles"]) == (76, 76, 0, 0)
    many = gp.gemm_plan(4096, 4096 + 2048, 1024, "i8", "row_col", 0, "pipelined", **kw)
    # 384 tiles leave 4 for a last wave: 8 half tiles
    assert (many["tiles"], many["dp_tiles"], many["half_tiles"]) == (384, 380, 4)
    over = gp.gemm_plan(4096, 4096 + 4096 + 2048, 1024, "i8", "row_col", 0, "pipelined", **kw)
    # 640 tiles leave 32 (at most 38) for a last wave
    assert (over["tiles"], over["half_tiles"]) == (640, 32)
    wide = gp.gemm_plan(4096, 4096 + 7 * 256, 1024, "i8", "row_col", 0, "pipelined", **kw)
    # 368 tiles leave 64 (more than half a wave): whole tiles only
    assert (wide["tiles"], wide["half_tiles"], wide["sk_tiles"]) == (368, 0, 0)
    f32 = gp.gemm_plan(1024, 1024, 1024, "f32", "row_row", 0, "pipelined", **kw)
    # 64 tiles: their K-loops dealt out as equal ranges to one CTA per SM (about 2.4 CTAs per
    # tile), two partial slots per CTA
    assert (f32["tiles"], f32["k_splits"], f32["grid"]) == (64, 3, 152)
    assert f32["workspace_bytes"] == 2 * 152 * 128 * 128 * 4
    # short K-loops: no range under 256 K steps (4 tiles x 1024 K = 16 ranges)
    small = gp.gemm_plan(256, 256, 1024, "f32", "row_row", 0, "pipelined", **kw)
    assert (small["tiles"], small["grid"], small["k_splits"]) == (4, 16, 4)
    # 80 tiles would keep 72 SMs idle: ranges as well (a tile shared by about two CTAs)
    half = gp.gemm_plan(1280, 1024, 2048, "f32", "row_row", 0, "pipelined", **kw)
    assert (half["tiles"], half["grid"], half["k_splits"]) == (80, 152, 2)
    f32_big = gp.gemm_plan(4096, 4096, 4096, "f32", "row_row", 0, "pipelined", **kw)
    # 1024 tiles leave the seventh wave part-empty: one range of the K-loops per SM (about 6.7
    # tiles each; a tile is shared by at most two CTAs)
    assert (f32_big["k_splits"], f32_big["grid"], f32_big["workspace_bytes"]) == (2, 152, 2 * 152 * 128 * 128 * 4)
    # whole waves, short K-loops, or nearly full single waves keep whole tiles
    for shape, tiles in (((4096, 4864, 1024), 1216), ((2048, 2048, 64), 256), ((1536, 1536, 2048), 144)):
        q = gp.gemm_plan(*shape, "f32", "row_row", 0, "pipelined", **kw)
        assert (q["tiles"], q["grid"], q["k_splits"], q["workspace_bytes"]) == (tiles, tiles, 1, 0), shape
    k256 = gp.gemm_plan(8192, 8192, 256, "bf16", "row_col", 0, "pipelined", **kw)
    # K <= 256: one CTA per 128 x 256 tile, persistent over the 152 SMs, whole tiles
    assert (k256["kernel"], k256["cta_pair"], k256["bn"], k256["stages"]) == ("umma_ring", 0, 256, 4)
    assert (k256["tiles"], k256["grid"], k256["sk_tiles"]) == (2048, 152, 0)
    assert gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined")["grid"] == 0   # no device queried
    with pytest.raises(gp.GemmError):
        gp.gemm_plan(4096, 4096, 4096, "f16", "row_col", 0, "pipelined", plan_sms=-1)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8", "f32"])
def test_plan_invariants_over_many_shapes(gp, dtype):
    # planned for a 152-SM GB300 without a device: whatever the shape and depth, the work split is
    # a partition of the tiles, the launch fits the SMs and shared memory, and each schedule's own
    # rules hold
    import itertools
    lay = "row_row" if dtype == "f32" else "row_col"
    sizes = (64, 128, 200, 520, 1000, 2048, 4104, 8192)
    ks = (16, 64, 128, 192, 256, 320, 1032, 4096, 16384)
    seen = set()
    for M, N, K in itertools.product(sizes, sizes, ks):
        if dtype == "f32" and K % 4:
            continue
        for S in (0, 2, 4, 6):
            rc = gp.gemm_plan_rc(M, N, K, dtype, lay, S, "pipelined")
            if rc != 0:
                continue
            p = gp.gemm_plan(M, N, K, dtype, lay, S, "pipelined", plan_sms=152)
            tiles, grid, dp, sk = p["tiles"], p["grid"], p["dp_tiles"], p["sk_tiles"]
            seen.update(k for k in ("b_resident", "half_tiles") if p[k])
            seen.update(["split after whole waves"] if sk and dp else ["split only"] if sk else [])
            seen.update(["k-split cluster"] if p["cta_pair"] == 3 else [])
            seen.update(["ffma ranges"] if p["k_splits"] > 1 else [])
            assert tiles == -(-M // p["bm"]) * -(-N // p["bn"]), (M, N, K, S)
            assert p["k_tiles"] == -(-K // p["bk"])
            assert 0 < grid <= 152 or (not p["persistent"] and grid == tiles)
            assert p["smem_bytes"] <= 232448 and 1 <= p["stages"] <= 8
            if dtype in ("f16", "bf16"):
                # whole tiles then split ones: the split tiles are the last, whole waves before them
                assert dp + sk == tiles and 0 <= sk
                workers = grid // (2 if p["cta_pair"] else 1)
                if sk:
                    assert p["cta_pair"] != 3 and p["workspace_bytes"] > 0
                    assert dp % workers == 0 and sk <= (2 if p["stages"] <= 4 else 1) * workers
                if p["b_resident"]:
                    assert (p["cta_pair"], sk) == (0, 0) and p["stages"] == p["k_tiles"] >= 2
                    assert tiles > grid and p["raster_gm"] == -(-M // p["bm"])
                if p["cta_pair"] == 3:
                    assert grid % 4 == 0 and tiles <= grid // 4
            elif dtype == "i8" and p["cta_pair"]:
                assert dp + sk + p["half_tiles"] == tiles or dp + sk == tiles
                assert not (sk and p["half_tiles"])
            elif dtype == "f32":
                assert p["k_splits"] >= 1 and (p["k_splits"] == 1) == (p["workspace_bytes"] == 0)
    # the sizes reach every schedule of the type
    want = {"f16": {"b_resident", "split after whole waves", "split only", "k-split cluster"},
            "bf16": {"b_resident", "split after whole waves", "split only", "k-split cluster"},
            "i8": {"half_tiles", "split only"}, "f32": {"ffma ranges"}}[dtype]
    assert want <= seen, want - seen
