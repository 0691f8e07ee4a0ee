"""Host-side pieces of bench.py, on the CPU: the FLOP convention, the clock
sampler's parsing of nvidia-smi lines, and the fallback peaks."""
import bench
import workloads


def test_flop_convention_of_the_benchmark_workload():
    w = workloads.WORKLOADS[bench.WORKLOAD]
    fwd, bwd = bench.flops(w)
    # causal: half of 4 B H Nq Nk d; the backward counts 2.5 times the forward
    assert fwd == 0.5 * 4 * w.B * w.H * w.Nq * w.Nk * w.d
    assert bwd == 2.5 * fwd
    assert abs(fwd - 2.75e11) / 2.75e11 < 0.01


def test_clock_summary_parses_reasons_and_skips_bad_lines():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "0, 2070, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1385.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = cs.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2010.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_slowdown():
    cs = bench.ClockSampler(0)
    cs.lines = ["0, 1500, 2070, 900.0, 0x40, Not Active, Active, Not Active, Not Active"]
    assert cs.summary()["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples_is_none():
    cs = bench.ClockSampler(0)
    cs.lines = []
    assert cs.summary() is None


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench.load_peaks()
    assert source == "fallback"
    assert peaks == bench.FALLBACK_PEAKS


def test_effective_flops_count_only_valid_keys():
    w = workloads.WORKLOADS["bf16_b8h16_q1024_k16384_d128_keypad"]
    lens = [w.Nk // 2] * w.B
    # half of the keys valid in every batch: half of the nominal count
    assert bench.effective_fwd_flops(w, lens) == 0.5 * bench.flops(w)[0]
    assert bench.effective_fwd_flops(w, None) == bench.flops(w)[0]


def test_both_arms_print_the_same_config():
    w = workloads.WORKLOADS[bench.WORKLOAD]
    assert bench.bench_config(w, 1) == bench.bench_config(w, 1)
    cfg = bench.bench_config(w, 1)
    assert cfg["workload"] == w.name and cfg["parallelism"] == "single GPU"
    assert bench.bench_config(w, 4)["parallelism"] == "replicas"
