"""Host-side logic of bench.py (CPU): the clock record taken during the timed
region, the per-launch DRAM traffic record that is only used while the kernel
sources still hash to the value it was taken with, and the peak denominators."""
import hashlib
import json
import os
import shutil

import bench


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clock_record_median_max_and_reasons(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1500, 2070, 1200.5, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "0, 1600, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "0, [N/A], 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "garbage line\n")
    cs = bench.ClockSampler(0)
    cs.proc, cs.path = _FakeProc(), str(path)
    rec = cs.stop()
    assert rec["sm_mhz"] == 1550.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 3 and rec["power_w_max"] == 1300.0
    assert not path.exists()


def test_clock_record_flags_thermal_reasons(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1400, 2070, 1400, 0x40, Active, Not Active, Active, Not Active\n")
    cs = bench.ClockSampler(0)
    cs.proc, cs.path = _FakeProc(), str(path)
    assert cs.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_record_is_dropped_when_a_kernel_source_changes(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic_tc_kernels_8b_vocab.json")))
    for src in rec["source_files"]:
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, src), dst)
    h = hashlib.sha256()
    for src in rec["source_files"]:
        h.update((tmp_path / src).read_bytes())
    rec["source_sha256"] = h.hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_tc_kernels_8b_vocab.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    name = next(iter(rec["kernels"]))
    k = rec["kernels"][name]
    assert bench.kernel_traffic(name) == k["dram_read_bytes"] + k["dram_write_bytes"]
    assert bench.kernel_traffic("no_such_kernel") is None
    src = tmp_path / rec["source_files"][-1]
    src.write_bytes(src.read_bytes() + b"\n// changed\n")
    assert bench.kernel_traffic(name) is None


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    burst, sustained, hbm, src = bench.measured_peaks()
    assert src == "fallback" and burst == bench.FALLBACK_BF16_TFLOPS and sustained == bench.FALLBACK_BF16_TFLOPS_SUSTAINED
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                                                              "hbm_gbs": 6600.0}))
    assert bench.measured_peaks() == (1900.0, 1700.0, 6600.0, "measured")
