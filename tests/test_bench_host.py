"""bench.py's host logic on the CPU: the clock record it attaches to every
line, the DRAM traffic it reads from the committed ncu summary only while the
kernel sources are unchanged, the peak it divides by, and the algorithmic
byte counts of the roofline."""
import json
import os

import pytest

import bench


def _clock_line(sm, smax, power, active="0x0", hw="Not Active", hw_th="Not Active", sw_th="Not Active",
                cap="Not Active"):
    return f"0, {sm}, {smax}, {power}, {active}, {hw}, {hw_th}, {sw_th}, {cap}\n"


def _summary(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(lines))
    c = bench.ClockSampler(0)
    c.path = str(path)
    c.proc = object()       # as if nvidia-smi had been started
    return c.summary()


def test_clock_summary_takes_the_loaded_half_and_collects_reasons(tmp_path):
    idle = [_clock_line(345, 2070, 150.0) for _ in range(4)]
    load = [_clock_line(2070, 2070, 900.0), _clock_line(2055, 2070, 950.0),
            _clock_line(2070, 2070, 1000.0, cap="Active"), _clock_line(2040, 2070, 980.0)]
    s = _summary(tmp_path, idle + load + ["garbage line\n", "0, [N/A], 2070, 1, x, y, z, w, v\n"])
    assert s["sm_mhz"] == pytest.approx(2062.5)     # median of the four loaded samples
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 8


def test_clock_summary_names_every_slowdown(tmp_path):
    lines = [_clock_line(1500, 2070, 800.0, hw="Active"), _clock_line(1400, 2070, 810.0, hw_th="Active"),
             _clock_line(1450, 2070, 820.0, sw_th="Active")]
    s = _summary(tmp_path, lines)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples(tmp_path):
    assert _summary(tmp_path, ["\n"])["reasons"] == ["no samples"]
    assert bench.ClockSampler(0).summary()["reasons"] == ["nvidia-smi unavailable"]


@pytest.fixture
def fake_csrc(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "a.cu").write_text("kernel a")
    (csrc / "b.cuh").write_text("kernel b")
    (csrc / "notes.txt").write_text("not a source")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(csrc / "a.cu"))
    return csrc


def test_kernel_source_hash_follows_every_source_file(fake_csrc):
    h0 = bench.kernel_source_sha()
    (fake_csrc / "notes.txt").write_text("changed")
    assert bench.kernel_source_sha() == h0            # only .cu and .cuh count
    (fake_csrc / "b.cuh").write_text("kernel b, changed")
    h1 = bench.kernel_source_sha()
    assert h1 != h0
    (fake_csrc / "c.cu").write_text("")
    assert bench.kernel_source_sha() != h1            # a new, even empty, source counts


def test_traffic_is_reported_only_for_the_profiled_sources(fake_csrc, tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    assert bench.stored_traffic("decode") is None     # no file
    path.write_text(json.dumps({"decode": {"kernel_source_sha": bench.kernel_source_sha(),
                                           "dram_bytes_per_launch": 18100000}}))
    assert bench.stored_traffic("decode") == 18100000
    assert bench.stored_traffic("prefill") is None    # not profiled
    (fake_csrc / "a.cu").write_text("kernel a, changed")
    assert bench.stored_traffic("decode") is None     # stale once a kernel changes
    path.write_text("{not json")
    assert bench.stored_traffic("decode") is None


def test_committed_traffic_entries_name_a_kernel_hash():
    with open(bench.TRAFFIC_PATH) as f:
        t = json.load(f)
    entries = {name: e for name, e in t.items() if not name.startswith("_")}
    assert entries, "no traffic entries"
    for name, e in entries.items():
        assert len(e["kernel_source_sha"]) == 16, name
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"] > 0, name
        assert "--clock-control none" in e["command"], name


def test_peak_falls_back_only_without_a_measurement(tmp_path, monkeypatch):
    path = tmp_path / "peaks.json"
    monkeypatch.setattr(bench, "PEAKS_PATH", str(path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    path.write_text(json.dumps({"hbm_gbs": 6759.9}))
    assert bench.hbm_peak() == (6759.9, "measured")


def test_algorithmic_bytes():
    # decode as built on a GPU: 64 rows summing to 4,494,799 scores, k = 2048
    assert bench.algorithmic_bytes(4_494_799, 64, 2048) == 18_503_996
    # prefill: L_i = max(1, (i + 1) // 4) over 16384 rows, k = 2048
    total = sum(max(1, (i + 1) // 4) for i in range(16384))
    assert total == 33_550_339
    assert bench.algorithmic_bytes(total, 16384, 2048) == 268_550_156
    # the statistics op writes 24 bytes per row instead of k indices
    assert bench.algorithmic_bytes_stats(4_494_799, 64) == 4 * 4_494_799 + 8 * 64 + 24 * 64


def test_warmup_below_three_is_refused(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--warmup", "2"])
    with pytest.raises(SystemExit, match="at least 3"):
        bench.main()


def test_single_process_reads_rank_zero(monkeypatch):
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert os.environ.get("RANK") is None
