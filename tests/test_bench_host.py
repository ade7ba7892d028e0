"""Host-side logic of bench.py that decides what a bench line reports: the
comment-insensitive kernel hash that keys the committed DRAM-traffic
figures, the traffic lookup that turns stale figures into null, the clock
record's parsing (its throttle reasons decide whether a run is rejected)
and the fallback peaks.  No GPU."""
import json
import os

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = "int a;  // the first\n\n/* a block\n   comment */ int b;\n  // only a comment\nint c;\n"
    assert bench._code_only(src) == "int a;\n int b;\nint c;"


def test_code_only_ignores_comment_edits_but_not_code_edits():
    base = "__global__ void k() {\n  // stage the tile\n  x = 1;\n}\n"
    reworded = "__global__ void k() {\n  // load the tile into shared memory\n  x = 1;  /* fast */\n}\n"
    changed = "__global__ void k() {\n  // stage the tile\n  x = 2;\n}\n"
    assert bench._code_only(base) == bench._code_only(reworded)
    assert bench._code_only(base) != bench._code_only(changed)


def _fake_tree(tmp_path, kernel_text):
    csrc = tmp_path / "fine_grained_fp8_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(kernel_text)
    (csrc / "fgq_device.cuh").write_text("// helpers\nint helper;\n")
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_is_null_once_the_kernel_code_changes(tmp_path, monkeypatch):
    csrc = _fake_tree(tmp_path, "int x = 1;  // v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench._kernel_sha("k.cu")
    table = {"kern": {"bytes_per_launch": 12345, "source": "k.cu", "source_sha": sha}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(table))
    assert bench._traffic("kern", "k.cu") == 12345
    # a comment edit keeps the capture
    (csrc / "k.cu").write_text("int x = 1;  // reworded\n")
    assert bench._traffic("kern", "k.cu") == 12345
    # a code edit retires it, and so does an edit of the shared device header
    (csrc / "k.cu").write_text("int x = 2;\n")
    assert bench._traffic("kern", "k.cu") is None
    (csrc / "k.cu").write_text("int x = 1;\n")
    assert bench._traffic("kern", "k.cu") == 12345
    (csrc / "fgq_device.cuh").write_text("int helper2;\n")
    assert bench._traffic("kern", "k.cu") is None
    # unknown kernels and a missing table give null, not an error
    assert bench._traffic("other", "k.cu") is None
    os.unlink(tmp_path / "profiles" / "traffic.json")
    assert bench._traffic("kern", "k.cu") is None


def _sampler_with(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(line + "\n" for line in lines))
    s = bench.ClockSampler(0)
    s.path = str(path)
    return s


def test_clock_summary_median_max_and_reasons(tmp_path):
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = [
        "0, 2070, 2070, 650.1, 0x0004, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 690.5, 0x0004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 600.0, 0x0000, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 610.0, 0x0000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    out = _sampler_with(tmp_path, lines).summary()
    assert out["samples"] == 4
    assert out["sm_mhz"] == 2070.0          # median of 2070, 1980, 2070 (the N/A row has none)
    assert out["sm_max_mhz"] == 2070.0
    assert out["power_w_max"] == 690.5
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_the_reasons_that_reject_a_run(tmp_path):
    lines = [
        "0, 1500, 2070, 700.0, 0x0008, Active, Not Active, Not Active, Not Active",
        "0, 1400, 2070, 700.0, 0x0040, Not Active, Active, Active, Not Active",
    ]
    out = _sampler_with(tmp_path, lines).summary()
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1450.0


def test_clock_summary_without_samples(tmp_path):
    out = _sampler_with(tmp_path, []).summary()
    assert out["samples"] == 0 and out["reasons"] == ["unsampled"]


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench._peaks()
    assert source == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6779.4, "bf16_tflops": 1921.4}))
    peaks, source = bench._peaks()
    assert source == "measured" and peaks["hbm_gbs"] == 6779.4
