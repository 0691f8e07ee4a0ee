"""Host-side pieces of bench.py, on the CPU: the FLOP convention, the clock
sampler's parsing of nvidia-smi lines, the fallback peaks, and the reference
arm's JSON line."""
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


def test_reference_arm_line_carries_the_contract_keys(monkeypatch, capsys):
    """The reference arm's JSON line (the oracle timed on the host cores):
    same metric, unit and config as the GPU arm, impl "reference", a
    cpu_baseline describing the run, and an e2e object with no copies. The
    oracle's timing is stubbed so that the test runs in no time."""
    import json
    import types
    monkeypatch.setattr(bench, "calibrated_oracle", lambda w, per_step: 8)
    monkeypatch.setattr(bench, "oracle_sample",
                        lambda w, n, seed_offset=0: (0.5, 2.0e9, "stub sample", 3))
    args = types.SimpleNamespace(steps=2, warmup=1, gpus=1)
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = workloads.WORKLOADS[bench.WORKLOAD]
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["config"] == bench.bench_config(w, 1)
    assert line["value"] == 2.0e9 / 0.5 / 1e12
    assert line["steps"] == 2 and line["warmup"] == 1 and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 3 and cb["value"] == line["value"]
    assert cb["sample"] == "stub sample"
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
