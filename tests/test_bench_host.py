"""Host-side logic of bench.py on the CPU: the byte counts behind every
GB/s figure, the ncu traffic record's validity check, the clock-record
parsing and the peak lookup.  No GPU."""
import os

import pytest

import bench
from precision_quantization_token_gb300.inputs import WORKLOADS


@pytest.mark.parametrize("name,total", [
    # read + codes + scales of the five casts, from the shapes: M*K*2 read
    # (M*2N*2 for SwiGLU), M*K (E4M3) or M*K/2 (E2M1) codes, and one fp32
    # scale (4 B) or UE8M0 byte per group
    ("c1", 256 * 1024 * 2 + 256 * 1024 + 256 * 8 * 4),
    ("c2", 4096 * 7168 * 2 + 4096 * 7168 + 4096 * 56),
    ("c3a", 16384 * 4096 * 2 + 16384 * 4096 + 16384 * 128 * 4),
    ("c3b", 16384 * 4096 * 2 + 16384 * 4096 + 16384 * 64 * 4),
    ("c4", 8192 * 4096 * 2 + 8192 * 2048 + 8192 * 16),
    ("c5", 32768 * 7168 * 2 + 32768 * 7168 // 2 + 32768 * 448),
])
def test_algorithmic_bytes(name, total):
    b = WORKLOADS[name].algorithmic_bytes()
    assert b["total"] == total == b["read"] + b["codes"] + b["scales"]


def test_algorithmic_bytes_match_the_published_table():
    """The totals the scope table prints for C1-C5."""
    want = {"c1": 794_624, "c2": 88_309_760, "c3a": 209_715_200,
            "c3b": 205_520_896, "c4": 84_017_152, "c5": 601_882_624}
    for name, total in want.items():
        assert WORKLOADS[name].algorithmic_bytes()["total"] == total, name


def _write_record(path, sha, workload="c2", nbytes=61_000_000):
    path.write_text("# test record\n"
                    f"workload: {workload}\n"
                    f"source_sha256: {sha}\n"
                    "dram_bytes_read: 1\ndram_bytes_write: 2\n"
                    f"dram_bytes_per_launch: {nbytes}\n")


def test_traffic_record_is_used_only_for_its_sources(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.txt"
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(rec))
    _write_record(rec, bench.kernel_source_hash())
    assert bench.profiled_traffic("c2") == 61_000_000
    assert bench.profiled_traffic("c3a") is None        # another workload
    _write_record(rec, "0" * 64)                        # sources changed since
    assert bench.profiled_traffic("c2") is None
    rec.write_text("garbage without fields\n")
    assert bench.profiled_traffic("c2") is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing"))
    assert bench.profiled_traffic("c2") is None


def test_source_hash_covers_the_kernel_sources(tmp_path, monkeypatch):
    """The hash changes when any hashed source changes."""
    root = tmp_path
    csrc = root / "precision_quantization_token_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "include").mkdir()
    for f in ("tk_cast.cu", "tk_device.cuh", "tk_internal.h"):
        (csrc / f).write_text(f)
    (root / "include" / "tk_cast.h").write_text("h")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    for f in ("tk_cast.cu", "tk_device.cuh", "tk_internal.h"):
        (csrc / f).write_text(f + " changed")
        assert bench.kernel_source_hash() != h0
        (csrc / f).write_text(f)
    (root / "include" / "tk_cast.h").write_text("h changed")
    assert bench.kernel_source_hash() != h0


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


class _DoneThread:
    def join(self, timeout=None):
        pass


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc, s.thread, s.lines = _DoneProc(), _DoneThread(), lines
    return s.stop()


def test_clock_record_parsing():
    ok = "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"
    slow = "0, 1500, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active"
    r = _sampler([ok, ok, capped])
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["power_w_max"] == 1400.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    r = _sampler([ok, slow, "garbled line", "0, N/A, 2070, 1, x, a, b, c, d"])
    assert r["samples"] == 2 and r["reasons"] == ["hw_slowdown"]
    assert r["sm_mhz"] == (2070.0 + 1500.0) / 2
    none = bench.ClockSampler(0).stop()
    assert none["sm_mhz"] is None and none["reasons"] == ["nvidia-smi unavailable"]


def test_peak_lookup(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6777.3}')
    assert bench.measured_peaks() == (6777.3, "measured (MEASURED_PEAKS.json hbm_gbs)")
    os.remove(tmp_path / "MEASURED_PEAKS.json")
    value, source = bench.measured_peaks()
    assert value == bench.FALLBACK_HBM_GBS and source.startswith("fallback")
