"""Host logic of bench.py that needs no GPU: the clock-sample summary, the ncu-summary
lookup behind the roofline's traffic figure, and the committed profile summaries."""
import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMI = """0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
0, 2025, 2070, 1350.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active
0, 2070, 2070, 1310.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
garbage line
"""


def test_clock_summary_parses_nvidia_smi_rows():
    c = bench.ClockSampler(0)
    c.text = SMI
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0          # median of 2070, 2025, 2070
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples():
    c = bench.ClockSampler(0)
    c.text = ""
    assert c.summary() is None


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    for kernel in ("spmma", "compress_meta"):
        (tmp_path / "profiles" / f"{kernel}_demo.txt").write_text(
            "# title\nsource_hash: abc123\ndram_bytes_per_launch: 4096\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda sources=bench.SPMMA_SOURCES: "abc123")
    assert bench.profile_traffic("demo") == 4096.0
    assert bench.profile_traffic("demo", "compress_meta") == 4096.0
    monkeypatch.setattr(bench, "source_hash", lambda sources=bench.SPMMA_SOURCES: "changed")
    assert bench.profile_traffic("demo") is None     # kernel changed since the capture
    assert bench.profile_traffic("demo", "compress_meta") is None
    assert bench.profile_traffic("missing") is None


def test_each_kernel_is_hashed_from_its_own_sources():
    assert "spmma.cu" in bench.SPMMA_SOURCES and "compress.cu" not in bench.SPMMA_SOURCES
    assert "compress.cu" in bench.COMPRESS_SOURCES and "spmma.cu" not in bench.COMPRESS_SOURCES
    assert bench.source_hash() != bench.source_hash(bench.COMPRESS_SOURCES)


def test_committed_gemm_profiles_name_their_command_and_counters():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "spmma_*.txt")))
    assert files
    for f in files:
        text = open(f).read()
        assert "# command: ncu " in text and "--clock-control none" in text
        fields = dict(line.split(":", 1) for line in text.splitlines()
                      if ":" in line and not line.startswith("#"))
        assert len(fields["source_hash"].strip()) == 16
        assert int(fields["dram_bytes_per_launch"]) > 0
