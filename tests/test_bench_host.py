"""Host logic of bench.py's reporting on CPU: the DRAM traffic read from committed ncu
summaries (gated by the hash of every kernel source they cover), the clock summary of the
nvidia-smi samples, and the fraction of the sustained peak."""
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# every committed summary bench.py reads, with the sources it names
SUMMARIES = [
    ("chunkwise_tc_pair_chunkwise_long.md", ("tc_chunkwise_pair.cu",)),
    ("chunkwise_backward_tc_backward.md", ("backward_tc.cu", "tc_chunkwise_pair.cu")),
    ("parallel_pair_parallel_norm.md", ("tc_parallel_pair.cu", "tc_parallel.cu")),
    ("decode_decode.md", ("decode.cu",)),
    ("rglru_scan_rglru.md", ("rglru.cu",)),
    ("xpos_kernel_xpos.md", ("xpos.cu",)),
    ("gemm_kernel_gemm.md", ("tc_gemm.cu",)),
]


@pytest.mark.parametrize("summary,sources", SUMMARIES)
def test_committed_summaries_match_the_current_sources(summary, sources):
    """A summary whose counters were taken on the current sources gives its bytes; the
    bench line would otherwise report traffic null."""
    got = bench.profile_traffic(summary, *sources)
    assert got is not None and got > 0, summary


def test_traffic_is_null_once_a_source_changes(tmp_path, monkeypatch):
    """The same summary against a kernel source whose text differs gives None."""
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "linear_recurrence_sequence_chunkwise_b300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copy(os.path.join(ROOT, "profiles", "decode_decode.md"), root / "profiles")
    src = os.path.join(ROOT, "linear_recurrence_sequence_chunkwise_b300", "csrc", "decode.cu")
    shutil.copy(src, csrc / "decode.cu")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.profile_traffic("decode_decode.md", "decode.cu") is not None
    with open(csrc / "decode.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.profile_traffic("decode_decode.md", "decode.cu") is None
    assert bench.profile_traffic("missing.md", "decode.cu") is None


def test_clock_summary_reads_reasons_and_loaded_samples(tmp_path):
    """Samples drawn under load set the median; every active throttle reason is listed."""
    c = bench.Clocks(0)
    c.path = str(tmp_path / "clocks.csv")
    rows = [
        "0, 2032, 2032, 120.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1850, 2032, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1870, 2032, 940.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2032, 2032, 125.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    with open(c.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    c.proc = object()          # as if the sampler had run
    s = c.summary()
    assert s["sm_mhz"] == 1870.0
    assert s["sm_max_mhz"] == 2032.0
    assert s["samples"] == 5 and s["samples_under_load"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 950.0
    assert not os.path.exists(c.path)


def test_sustained_fraction():
    assert bench.sustained_frac(1384.1, {"bf16_tflops_sustained": 1384.1}) == {
        "peak_sustained": 1384.1, "frac_of_sustained": 1.0}
    assert bench.sustained_frac(1000.0, {"bf16_tflops": 1762.3}) == {}
