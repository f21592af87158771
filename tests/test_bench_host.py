"""The benchmark's host side on CPU: compulsory bytes and FLOPs behind the
roofline figures, the clock-record summary, the peaks file, the rule that a
DRAM-traffic record counts only at the sources it was taken on, and the
reference arm's JSON line (the oracle timed on the host)."""
import os

import pytest

import bench
import synth


# (workload, token-heads, compulsory MB, GFLOP), worked out from the counting
# rule: (2 d_k + 2 d_v) * io bytes + 8 bytes of gates per token-head, h0 read
# and hT written once per (sequence, head); 6 C d_k + 4 C d_v + 6 d_k d_v FLOPs
# per token-head with C = 64
FORWARD_CASES = [
    ("gdn_fwd_b1_h1_t256_d64_fp32", 256, 0.2806, 0.01678),
    ("gdn_fwd_b4_h16_t4096_d128_bf16", 262144, 274.7, 47.24),
    ("gdn_fwd_b8_h8_t8192_d64_bf16_h0", 524288, 274.7, 34.36),
    ("gdn_fwd_b1_h16_t131072_d128_bf16", 2097152, 2165.3, 377.96),
]


@pytest.mark.parametrize("name,tokens,mb,gflop", FORWARD_CASES)
def test_forward_compulsory_bytes_and_flops(name, tokens, mb, gflop):
    shape = bench.workload_shape(name)
    assert shape["tokens"] == tokens
    by, fl = bench.algorithmic(shape)
    assert abs(by / 1e6 - mb) <= 5e-4 * mb
    assert abs(fl / 1e9 - gflop) <= 5e-4 * gflop


def test_default_workload_bytes_by_hand():
    # 262 144 token-heads x 1032 bytes, plus hT: 64 heads x 128 x 128 x 4 bytes
    by, _ = bench.algorithmic(bench.workload_shape(bench.DEFAULT_WORKLOAD))
    assert by == 262144 * (2 * 128 * 2 + 2 * 128 * 2 + 8) + 64 * 128 * 128 * 4


def test_varlen_counts_follow_the_drawn_lengths():
    name = "gdn_fwd_varlen_n64_h32_dk128_dv256_bf16"
    cfg = synth.WORKLOADS[name]
    lens = synth.varlen_lengths(cfg["N"], cfg["len_min"], cfg["len_max"], cfg["seed"])
    shape = bench.workload_shape(name)
    assert shape["tokens"] == int(lens.sum()) * 32
    by, fl = bench.algorithmic(shape)
    assert fl == shape["tokens"] * 311296          # 6*64*128 + 4*64*256 + 6*128*256
    state = 64 * 32 * 256 * 128 * 4
    assert by == shape["tokens"] * ((2 * 128 + 2 * 256) * 2 + 8) + 2 * state


def test_decode_bytes_are_the_state_round_trip():
    shape = bench.workload_shape("gdn_decode_b256_h32_d128_bf16")
    by, fl = bench.algorithmic(shape)
    th = 256 * 32
    assert by == th * ((2 * 128 + 2 * 128) * 2 + 8 + 2 * 128 * 128 * 4)
    assert fl == th * 6 * 128 * 128


def test_single_process_reduction_and_throughput():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    # 1000 token-heads in 2 ms on each of 4 replicas
    assert bench.job_throughput(1000, 4, 2.0) == pytest.approx(2e6)


def test_clock_summary_takes_the_loaded_samples_and_reasons():
    s = bench.ClockSampler(0)
    s.lines = [
        "0, 1000, 2070, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    out = s.summary()
    # the idle sample (below half the maximum) is left out of the median
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 4
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unavailable"]


def test_peaks_fall_back_when_the_file_is_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    hbm, tf, kind = bench.load_peaks()
    assert kind == "fallback" and hbm == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000.5, "bf16_tflops": 1800}')
    assert bench.load_peaks() == (7000.5, 1800.0, "measured")


def test_traffic_record_counts_only_at_its_own_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "gated_deltanet_recurrence_gdn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (tmp_path / "include" / "gdn.h").write_text("/* header */\n")
    (csrc / "k.cu").write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k_x": ["k.cu"]})
    assert bench.recorded_traffic("k_x", "w") is None          # no record file yet
    h = bench.kernel_source_hash("k_x")
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel workload source_hash bytes\nk_x w %s 123456\nk_x other %s 7\n" % (h, h))
    assert bench.recorded_traffic("k_x", "w") == 123456.0
    assert bench.recorded_traffic("k_y", "w") is None          # another kernel
    (csrc / "k.cu").write_text("// kernel v2\n")               # sources changed
    assert bench.recorded_traffic("k_x", "w") is None
    (csrc / "k.cu").write_text("// kernel v1\n")
    (tmp_path / "include" / "gdn.h").write_text("/* header, edited */\n")
    assert bench.recorded_traffic("k_x", "w") is None          # the header counts too


def test_every_timed_kernel_names_existing_sources():
    csrc = os.path.join(bench.ROOT, "gated_deltanet_recurrence_gdn_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)


def test_reference_arm_line_keeps_the_contract():
    # the oracle timed on the host cores, on a bounded sample (rank 0 only)
    args = type("A", (), {"workload": "gdn_fwd_b1_h1_t256_d64_fp32", "steps": 1,
                          "warmup": 0, "cpu_seconds": 1.0})()
    assert bench.run_reference(args, 2, 1) is None          # other ranks: no work
    line = bench.run_reference(args, 1, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["metric"] == bench.METRIC and line["dtype"] == "f64"
    assert line["config"]["workload"] == "gdn_fwd_b1_h1_t256_d64_fp32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert cb["unit"] == line["unit"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["steps"] == 1 and line["warmup"] == 0 and line["n_gpus"] == 1
