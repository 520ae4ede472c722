"""The benchmark's host-side bookkeeping on CPU: the roofline figures, the clock and
throttle summary, the gate that reports DRAM traffic only for the kernel sources it was
captured on, and the JSON line of both arms.  No GPU and no nvidia-smi: the clock
samples are written here, and the GPU leg of the library arm is replaced by its result
record."""
import json
import os

import pytest

import bench
import workloads

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}


def test_tensor_bound_roofline_takes_burst_or_sustained_peak():
    w = workloads.WORKLOADS["gemm_relu_1024_f16_128x128x64s3"]
    assert w.flops == 2 * 1024 ** 3
    r = bench.roofline(w, 0.01, PEAKS, "measured", {"reasons": []}, attn=False)
    achieved = 2 * 1024 ** 3 / 1e-5 / 1e12
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(achieved, abs=0.05)
    assert r["peak"] == 2000.0 and r["frac"] == pytest.approx(achieved / 2000.0, abs=1e-4)
    assert "burst" in r["peak_source"]
    capped = bench.roofline(w, 0.01, PEAKS, "measured", {"reasons": ["sw_power_cap"]}, False)
    assert capped["peak"] == 1600.0
    assert capped["frac"] == pytest.approx(achieved / 1600.0, abs=1e-4)
    assert capped["frac_of_burst"] == pytest.approx(achieved / 2000.0, abs=1e-4)
    assert "power cap" in capped["peak_source"]
    # no clock record at all: the burst peak
    assert bench.roofline(w, 0.01, PEAKS, "fallback", None, False)["peak"] == 2000.0


def test_eight_bit_operands_double_the_tensor_peak():
    w = workloads.WORKLOADS["gemm_8192_e4m3_tb"]
    r = bench.roofline(w, 1.0, PEAKS, "measured", {"reasons": []}, attn=False)
    assert r["peak"] == 2 * 2000.0 and "8-bit" in r["peak_source"]
    assert r["frac"] == pytest.approx(w.flops / 1e-3 / 1e12 / 4000.0, abs=1e-4)


def test_skinny_product_is_measured_against_memory_bandwidth():
    w = workloads.WORKLOADS["gemm_m16_n8192_k8192_bf16"]
    # 16 x 8192 x 8192: about 16 flops per byte, far under the ridge point (~333 here)
    assert w.flops / w.bytes_moved < PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    assert bench.is_hbm_bound(w, PEAKS)
    assert not bench.is_hbm_bound(workloads.WORKLOADS["gemm_8192_bf16_tb"], PEAKS)
    r = bench.roofline(w, 0.025, PEAKS, "measured", {"reasons": ["sw_power_cap"]}, False)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(w.bytes_moved / 2.5e-5 / 1e9, abs=0.05)
    assert "frac_of_burst" not in r


def test_attention_is_always_a_contraction():
    w = workloads.ATTN_WORKLOADS["attn_fwd_b4_h32_s4096_d128_bf16"]
    r = bench.roofline(w, 1.0, PEAKS, "measured", {"reasons": []}, attn=True)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0


def test_graph_chunks_cover_every_step_once_and_keep_the_rotation():
    for steps, rot in [(20, 1), (20, 42), (3, 1), (7, 2), (1000, 42), (5000, 42), (9000, 1)]:
        chunks = bench.graph_chunks(steps, rot)
        covered = [i for first, n, _ in chunks for i in range(first, first + n)]
        assert covered == list(range(steps)), (steps, rot)
        for first, n, reuse in chunks:
            if reuse:                       # a replay of the first graph: same sets in order
                assert first % rot == 0 and n == chunks[0][1] and chunks[0][0] == 0
    # up to 4096 steps: one graph, no graph boundary between timed calls
    assert bench.graph_chunks(20, 1) == [(0, 20, False)]
    assert bench.graph_chunks(4096, 42) == [(0, 4096, False)]
    # more steps: one graph of a whole number of rotations, replayed, then the rest
    ch = bench.graph_chunks(5000, 42)
    assert ch[0] == (0, 84, False) and all(c[1] == 84 and c[2] for c in ch[1:-1])
    assert ch[-1] == (59 * 84, 5000 - 59 * 84, False)
    assert bench.graph_chunks(0, 3) == []


def test_spread_takes_percentiles_over_equal_chunks():
    assert bench.percentile([1.0, 2.0, 3.0, 4.0, 5.0], 50) == 3.0
    assert bench.percentile([1.0, 2.0, 3.0, 4.0, 5.0], 10) == pytest.approx(1.4)
    assert bench.percentile([7.0], 90) == 7.0
    chunks = [(0, 4, False), (4, 4, False), (8, 4, False), (12, 4, False), (16, 4, False),
              (20, 2, False)]
    sp = bench.spread_of([4.0, 4.4, 4.0, 3.6, 4.8, 100.0], chunks)
    # the short remainder chunk is left out; per-call times are ms / 4
    assert sp["chunks"] == 5 and sp["calls_per_chunk"] == 4
    m = sp["ms_per_call"]
    assert m["min"] == pytest.approx(0.9) and m["max"] == pytest.approx(1.2)
    assert m["p50"] == pytest.approx(1.0) and m["p10"] <= m["p50"] <= m["p90"]


def test_nvml_samples_are_summarised_like_the_nvidia_smi_ones():
    # reason bits of the NVML clock-event mask
    assert bench.nvml_reason_names(0x4) == {"sw_power_cap"}
    assert bench.nvml_reason_names(0x1 | 0x8 | 0x40) == {"hw_slowdown", "hw_thermal_slowdown"}
    assert bench.nvml_reason_names(0x20) == {"sw_thermal_slowdown"}
    s = bench.summarise_samples([(1500.0, 2070.0, 1390.0, {"sw_power_cap"}),
                                 (1470.0, 2070.0, 1397.0, set()), (1485.0, None, None, set())])
    assert s["sm_mhz"] == 1485.0 and s["sm_max_mhz"] == 2070.0 and s["power_w_max"] == 1397.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    assert bench.summarise_samples([])["reasons"] == ["no samples"]


def test_short_timed_regions_borrow_the_last_pre_heat_samples():
    times = [0.0, 1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0]      # seconds
    # a long region keeps its own samples only
    idx, n, lead = bench.clock_window(times, 0.5, 2.5, 7.5, 5)
    assert idx == [3, 4, 5, 6, 7] and n == 5 and lead == 0.0
    # a short one is made up to five samples from the pre-heat right before it
    idx, n, lead = bench.clock_window(times, 0.5, 5.5, 6.5, 5)
    assert idx == [2, 3, 4, 5, 6] and n == 1 and lead == pytest.approx(3500.0)
    # never from before the pre-heat started
    idx, n, lead = bench.clock_window(times, 3.5, 5.5, 6.5, 5)
    assert idx == [4, 5, 6] and n == 1
    # no pre-heat mark: the region alone, however short
    idx, n, lead = bench.clock_window(times, None, 5.5, 6.5, 5)
    assert idx == [6] and n == 1 and lead == 0.0


def _row(sm, power, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return ", ".join(["0", str(sm), "2070", str(power), "0x0"] + flags) + "\n"


def test_clock_summary_takes_the_median_of_busy_samples_and_every_reason_seen():
    lines = [_row(345, 110.0), _row(2070, 800.0), _row(1890, 1390.5, ["sw_power_cap"]),
             _row(1950, 1200.0), "garbage line\n", "0, [N/A], 2070, 5, 0x0, a, b, c, d\n",
             _row(2070, 900.0)]
    c = bench.summarise_clocks(lines)
    # the idle 345 MHz sample is under half the highest and is left out of the median
    assert c["sm_mhz"] == pytest.approx(2010.0)
    assert c["sm_max_mhz"] == 2070.0 and c["power_w_max"] == 1390.5
    assert c["samples"] == 5 and c["reasons"] == ["sw_power_cap"]
    hot = bench.summarise_clocks([_row(1200, 700.0, ["hw_thermal_slowdown", "hw_slowdown"])])
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.summarise_clocks([])["reasons"] == ["no samples"]


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        table = json.load(f)
    name = "gemm_relu_1024_f16_128x128x64s3"
    entry = table[name]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: entry["kernel_source_hash"])
    assert bench.load_traffic(name) == entry["dram_bytes_per_launch"]
    assert bench.load_traffic("no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.load_traffic(name) is None


def test_source_hash_covers_every_kernel_source():
    for rel in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(bench.ROOT, rel)), rel
    csrc = os.path.join(bench.ROOT, "tiled_gemm_gb300", "csrc")
    kernels = {f"tiled_gemm_gb300/csrc/{f}" for f in os.listdir(csrc)
               if f.endswith((".cu", ".cuh"))}
    assert kernels <= set(bench.KERNEL_SOURCES)


CONTRACT_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                 "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                 "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"}


def _main_line(monkeypatch, capsys, argv):
    monkeypatch.setattr("sys.argv", ["bench.py"] + argv)
    bench.main()
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1
    return json.loads(out[0])


def test_json_line_of_the_library_arm(monkeypatch, capsys):
    # the GPU leg replaced by its result record: 10 steps of 0.01 ms each
    import torch
    monkeypatch.setattr(torch.cuda, "set_device", lambda *_: None)
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    spread = bench.spread_of([0.05, 0.052], [(0, 5, False), (5, 5, False)])
    fake = {"total_ms": 0.1, "rotation_sets": 42, "launches_per_step": 1, "clocks": clocks,
            "spread": spread, "plan": {"bm": 128},
            "e2e": {"value": 50.0, "unit": "TFLOP/s", "h2d_bytes_per_step": 4 << 20,
                    "d2h_bytes_per_step": 2 << 20}}
    monkeypatch.setattr(bench, "run_tl", lambda *a: fake)
    name = "gemm_relu_1024_f16_128x128x64s3"
    d = _main_line(monkeypatch, capsys, ["--steps", "10", "--warmup", "3", "--no-cpu-baseline",
                                         "--workload", name])
    assert CONTRACT_KEYS <= set(d)
    w = workloads.WORKLOADS[name]
    assert d["config"]["workload"] == name and d["n_gpus"] == 1
    assert d["value"] == pytest.approx(w.flops * 10 / 1e-4 / 1e12, rel=1e-4)
    assert d["higher_is_better"] is True and d["vs_baseline"] is None and d["dtype"] == "f16"
    assert d["gpu_launches"] == 10 and d["clocks"] == clocks
    assert d["roofline"]["bound"] == "tensor" and d["roofline"]["kernel_ms"] == 0.01
    assert d["roofline"]["algorithmic"]["flops_per_launch"] == w.flops
    assert "42 sets" in d["config"]["l2"]
    # the spread: per-call time of each chunk, and the rate at each
    sp = d["spread"]
    assert sp["chunks"] == 2 and sp["ms_per_call"]["min"] == pytest.approx(0.01)
    assert sp["ms_per_call"]["max"] == pytest.approx(0.0104)
    assert sp["tflops"]["min"] == pytest.approx(w.flops / 1e-5 / 1e12, abs=0.1)


def test_default_workload_is_the_largest_square_product(monkeypatch, capsys):
    # the bench's default is 8192^3 bf16 with a column-major B: the workload the
    # tensor-peak fraction is stated for
    import torch
    monkeypatch.setattr(torch.cuda, "set_device", lambda *_: None)
    assert workloads.HEADLINE == "gemm_8192_bf16_tb"
    fake = {"total_ms": 14.0, "rotation_sets": 1, "launches_per_step": 1,
            "clocks": {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]},
            "plan": {}, "e2e": None}
    monkeypatch.setattr(bench, "run_tl", lambda *a: fake)
    d = _main_line(monkeypatch, capsys, ["--steps", "20", "--warmup", "5", "--no-cpu-baseline"])
    w = workloads.WORKLOADS["gemm_8192_bf16_tb"]
    assert d["config"]["workload"] == "gemm_8192_bf16_tb" and d["dtype"] == "bf16"
    assert (w.M, w.N, w.K, w.trans_b) == (8192, 8192, 8192, True)
    assert d["config"]["l2"] == "operands larger than 2x L2"
    assert d["value"] == pytest.approx(w.flops * 20 / 14e-3 / 1e12, rel=1e-4)
    # under the power cap the roofline takes the sustained peak
    assert d["roofline"]["peak_source"].startswith("measured (sustained")
    assert d["roofline"]["frac"] == pytest.approx(d["roofline"]["achieved"] /
                                                  d["roofline"]["peak"], abs=1e-3)


def test_cpu_baseline_runs_the_oracle_on_all_cores_and_on_one(monkeypatch, capsys):
    # the real oracle on the host cores for a tiny budget, the GPU leg stubbed as above
    import torch
    monkeypatch.setattr(torch.cuda, "set_device", lambda *_: None)
    fake = {"total_ms": 0.1, "rotation_sets": 42, "launches_per_step": 1,
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
            "plan": {}, "e2e": None}
    monkeypatch.setattr(bench, "run_tl", lambda *a: fake)
    name = "gemm_relu_1024_f16_128x128x64s3"
    d = _main_line(monkeypatch, capsys, ["--steps", "10", "--warmup", "3",
                                         "--cpu-budget-s", "0.2", "--workload", name])
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == (os.cpu_count() or 1)
    assert cpu["value"] > 0 and "GFLOP" in cpu["sample"]
    one = cpu["single_core"]
    assert one["value"] > 0 and one["unit"] == "TFLOP/s"
    w = workloads.WORKLOADS[name]
    # the rate keeps 4 significant figures, the time one decimal
    assert one["workload_s"] == pytest.approx(w.flops / (one["value"] * 1e12), rel=1e-3, abs=0.1)
    assert bench.sig4(4.6449e-05) == 4.645e-05 and bench.sig4(1234.56) == 1235.0


def test_json_line_of_the_reference_arm(monkeypatch, capsys):
    # the oracle's timing replaced by a fixed rate: the line carries the arm's own keys
    monkeypatch.setattr(bench, "oracle_rate",
                        lambda w, a, b, budget, threads: (0.004, 0.5, 2e9, 64, 3))
    d = _main_line(monkeypatch, capsys, ["--impl", "reference", "--steps", "2",
                                         "--warmup", "3"])
    # both arms name the same configuration, rotation note included
    assert d["config"]["l2"] == "operands larger than 2x L2"
    assert d["impl"] == "reference" and d["value"] == 0.004 and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == 0.004
    assert d["e2e"] == {"value": 0.004, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == workloads.HEADLINE


def test_warmup_below_three_is_refused(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.main()
