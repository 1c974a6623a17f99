"""Host-side logic of the benchmark, on the CPU: which roof bounds each workload,
the algorithmic bytes per GEMM, and the replicas' max-over-ranks timing run as
two gloo processes."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from software_pipelined_tiled_pipeline_gb300.workloads import WORKLOADS

PEAKS = {"hbm_gbs": 6780.0, "bf16_tflops": 1920.5, "bf16_tflops_sustained": 1716.2}


def test_algorithmic_bytes():
    # A + B read once, C written once
    assert WORKLOADS["f16_4096"].algorithmic_bytes == 3 * 4096 * 4096 * 2
    assert WORKLOADS["i8_4096"].algorithmic_bytes == 2 * 4096 * 4096 + 4096 * 4096 * 4
    assert WORKLOADS["f32_1024"].algorithmic_bytes == 3 * 1024 * 1024 * 4
    assert WORKLOADS["bf16_8192_k256"].algorithmic_bytes == 2 * 8192 * 256 * 2 + 8192 * 8192 * 2
    assert WORKLOADS["bf16_skinny"].algorithmic_bytes == (8192 + 128) * 8192 * 2 + 8192 * 128 * 2


@pytest.mark.parametrize("name,kernel,bound", [
    ("f16_4096", "umma_pair_ring", "tensor"),
    ("i8_4096", "umma_i8_pair_ring", "tensor"),
    ("f32_1024", "ffma_ring", "alu"),
    ("bf16_8192_k256", "umma_pair_ring", "hbm"),     # the 128 MiB C write outweighs 34 GFLOP
    ("bf16_8192_k1024", "umma_pair_ring", "tensor"),
    ("bf16_8192_k16384", "umma_pair_ring", "tensor"),
    ("bf16_skinny", "umma_ring", "hbm"),             # the 128 MiB A read outweighs 17 GFLOP
])
def test_roofline_bound(name, kernel, bound):
    w = WORKLOADS[name]
    b, frac = bench.roofline_row(w, kernel, 1.0, PEAKS, 158.4)
    assert b == bound
    # a launch that takes exactly the roof's time is at fraction 1
    t_roof = max(w.ops / (bench.compute_peak(kernel, PEAKS, 158.4) * 1e12), w.algorithmic_bytes / (6780.0 * 1e9))
    assert bench.roofline_row(w, kernel, t_roof * 1e3, PEAKS, 158.4)[1] == pytest.approx(1.0, abs=1e-4)


def test_read_write_roof_takes_the_slowest_stream():
    rw = {"copy_gbs": 6800.0, "read_gbs": 6300.0, "write_gbs": 4000.0}
    w = WORKLOADS["bf16_8192_k256"]          # 8 MB read, 134 MB written: the write stream bounds it
    assert bench.rw_roof_us(w, rw) == pytest.approx(w.write_bytes / 4000.0 / 1e3)
    w = WORKLOADS["bf16_skinny"]             # 138 MB read, 2 MB written: the read stream bounds it
    assert bench.rw_roof_us(w, rw) == pytest.approx(w.read_bytes / 6300.0 / 1e3)
    assert w.read_bytes + w.write_bytes == w.algorithmic_bytes


def test_imma_rows_use_the_imma_ceiling():
    w = WORKLOADS["i8_4096"]
    _, frac = bench.roofline_row(w, "imma_ring", w.ops / 158.4e12 * 1e3 * 2, PEAKS, 158.4)
    assert frac == pytest.approx(0.5, abs=1e-4)


def test_job_throughput_counts_every_rank():
    # 4 ranks, 10 steps of 2*4096^3 each in 1 ms
    assert bench.job_throughput(2 * 4096 ** 3, 4, 10, 1.0) == pytest.approx(4 * 10 * 2 * 4096 ** 3 / 1e-3 / 1e12)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        total = bench.max_over_ranks(torch, dist, my_ms, "cpu")
        value = bench.job_throughput(1e12, world, 3, total)
        with open(os.path.join(outdir, "r%d.json" % rank), "w") as f:
            json.dump({"total": total, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("r%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["total"] == 15.0
        assert r["value"] == pytest.approx(1e12 * 2 * 3 / 15e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(torch, None, 7.5, "cpu") == 7.5


def test_capture_records_follow_code_not_comments():
    # a recorded ncu capture stays valid across comment edits and goes stale on code edits
    src = "int f(int x) {  // twice\n  return 2 * x; /* doubled */\n}\n"
    same = "int f(int x) {\n  // a new remark\n  return 2 * x;\n}\n"
    other = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)


def test_traffic_records_are_well_formed():
    # every committed DRAM-traffic record carries its read and write bytes and the hash of the
    # kernel code it was taken on (the bench reports the traffic only while that hash matches)
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "traffic.json")
    records = json.load(open(path))
    assert records
    for key, rec in records.items():
        assert rec["dram_bytes_per_launch"] == rec["dram_read"] + rec["dram_write"] > 0, key
        assert len(rec["source_sha"]) == 16 and int(rec["source_sha"], 16) >= 0, key
        assert os.path.exists(os.path.join(os.path.dirname(path), os.path.basename(rec["capture"]))), key


def test_final_line_fits_the_driver_tail():
    # a line as large as the bench builds it stays under 2 KB: optional keys go, required ones stay
    line = {"metric": bench.METRIC, "value": 1690.12, "unit": "TFLOPS", "n_gpus": 1, "steps": 20, "warmup": 5,
            "ms_per_step": 0.08134, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": "f16_4096", "M": 4096, "N": 4096, "K": 4096, "layout": "row_col",
                       "variant": "pipelined", "stages": 5, "kernel": "umma_pair_ring", "tile": "256x256x64",
                       "grid": 152, "l2": "inputs and output rotated over 4 buffer sets (384 MiB > 129 MB L2)",
                       "parallelism": "single"},
            "roofline": {"kernel": "umma_pair_ring", "kernel_avg_ms": 0.08134, "launch_isolated_ms": 0.0851,
                         "traffic": 144812345, "bound": "tensor", "achieved": 1690.12, "peak": 1920.5,
                         "unit": "TFLOP/s", "frac": 0.88,
                         "peak_source": "measured (MEASURED_PEAKS.json): dense bf16 burst (FP16 at the same rate)"},
            "e2e": {"value": 372.1, "unit": "TFLOPS", "h2d_bytes_per_step": 67108864, "d2h_bytes_per_step": 33554432},
            "gpu_launches": 20, "clocks": {"sm_mhz": 1560.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                                           "samples": 33},
            "library_same_shape": {"value": 1760.2, "ours_over_library": 0.951},
            "sustained": {"value": 1455.2, "frac": 0.848, "seconds": 3.01, "sm_mhz": 1540.0},
            "int8_4096": {"TOPS": 1398.2, "frac": 0.728, "stages": 6, "kernel": "umma_i8_pair_ring",
                          "launches_per_call": 2, "imma_ring_TOPS": 147.6, "imma_ceiling": 158.2},
            "int8_4096_inputs_ready": {"TOPS": 1430.1, "frac": 0.745, "caller_promise": True},
            "f16_stages": {"2": 979.1, "3": 1384.2, "4": 1551.3, "5": 1649.1, "6": 1645.2, "pingpong": 495.1},
            "f16_best_stage": 5, "pipelining_gain_like_for_like": {"f16_ring_s2_over_pingpong": 1.512},
            "fp32_1024": {"TFLOPS": 41.8, "frac_alu": 0.5193, "s2_over_pingpong": 1.79, "pingpong_TFLOPS": 23.3},
            "cpu_baseline": {"value": 0.044698, "unit": "TFLOPS", "cores": 16, "kind": "oracle",
                             "sample": "first 512 of 4096 rows of C in 10.1 s"},
            "sweep_file": "bench_sweep.json"}
    out = bench.compact_line(dict(line))
    assert len(json.dumps(out)) < 2000
    for k in ("metric", "value", "unit", "roofline", "e2e", "cpu_baseline", "clocks", "config", "gpu_launches"):
        assert k in out
    big = dict(line, padding="x" * 3000)
    out = bench.compact_line(big)
    assert len(json.dumps(out)) < 2000 and "padding" not in out and "roofline" in out
