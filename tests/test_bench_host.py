"""Host-side logic of bench.py: the algorithmic bytes and flops behind the
roofline, the comment-insensitive kernel-source hash that guards the ncu
traffic record, the clock-sample window and small parsers.  CPU only."""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = argv
    return b


def test_algorithmic_bytes_and_flops(bench):
    import workloads as wl
    w = wl.Workload("t", 9, T=10, H=256, E=4, k=2, I=128, R=2, ranks_per_node=2)
    counts = np.array([5, 0, 7, 8])            # 3 active experts, A = 20
    a = bench.algorithmic(w, counts, np.arange(4))
    A, T, H, I = 20, 10, 256, 128
    wb = 3 * 6 * H * I
    assert a["permute"]["bytes"] == T * H * 2 + A * H * 2
    assert a["grouped_ffn"]["flops"] == 6 * A * H * I
    assert a["grouped_ffn"]["weight_bytes"] == wb
    assert a["grouped_ffn"]["bytes"] == wb + A * H * 2 + A * I * 4 + A * H * 2
    assert a["combine"]["bytes"] == A * H * 2 + T * H * 2 + A * 8
    # the gather-fused FFN reads token rows instead of dispatched rows
    g = bench.algorithmic(w, counts, np.arange(4), gather=True)
    assert a["grouped_ffn"]["bytes"] - g["grouped_ffn"]["bytes"] == (A - T) * H * 2
    # FP8 dispatch: H code bytes + one fp32 scale per 128 channels per row
    f = bench.algorithmic(w, counts, np.arange(4), fp8=True)
    assert f["permute"]["bytes"] == T * H * 2 + A * (H + 4 * (H // 128))
    assert f["dequant"]["bytes"] == A * (H + 4 * (H // 128)) + A * H * 2
    # drops: only kept assignments run
    d = bench.algorithmic(w, counts, np.arange(4), kept=15)
    assert d["grouped_ffn"]["flops"] == 6 * 15 * H * I


def test_algorithmic_shared_expert_separate_or_fused(bench):
    import workloads as wl
    w = wl.Workload("s", 9, T=10, H=256, E=4, k=2, I=128, R=2, ranks_per_node=2, shared_I=128)
    counts = np.array([5, 5, 5, 5])
    sep = bench.algorithmic(w, counts, np.arange(4))
    fus = bench.algorithmic(w, counts, np.arange(4), fused_shared=True)
    assert "shared_ffn" in sep and "shared_ffn" not in fus
    for key in ("flops", "weight_bytes", "bytes"):
        assert fus["grouped_ffn"][key] == sep["grouped_ffn"][key] + sep["shared_ffn"][key]
    assert fus["permute"]["bytes"] == sep["permute"]["bytes"] + 10 * 256 * 2
    # the combine also reads the shared output either way
    assert fus["combine"]["bytes"] == sep["combine"]["bytes"]


def test_kernel_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// header\nint f(int x) { return x + 1; }  /* note */\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(src)])
    h0 = bench.kernel_source_hash()
    src.write_text("// a different header\n\nint f(int x) {\n  return x + 1;  // same code\n}\n")
    assert bench.kernel_source_hash() == h0
    src.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_clock_summary_keeps_the_timed_window(bench):
    cs = bench.ClockSampler(0)
    line = lambda mhz, cap: f"0, {mhz}, 2070, 900, 0x0, Not Active, Not Active, Not Active, {cap}"
    cs.lines = [(1.00, line(2070, "Not Active")),      # before the region
                (2.00, line(1500, "Active")),          # inside
                (2.01, line(1600, "Not Active")),      # inside
                (3.00, line(1000, "Active"))]          # after
    s = cs.summary(1.5, 2.5)
    assert s["samples"] == 2 and s["sm_mhz"] == 1550.0 and s["reasons"] == ["sw_power_cap"]
    first = cs.summary(1.5, None, first=1)
    assert first["samples"] == 1 and first["sm_mhz"] == 1500.0
    assert cs.summary(5.0, 6.0)["samples"] == 0


def test_parse_relax(bench):
    assert bench.parse_relax("") is None
    assert bench.parse_relax("1/10") == (1, 10)
    assert bench.parse_relax("2") == (2, 1)


def test_tensor_peak_follows_the_timed_region_clocks(bench):
    peaks = {"bf16_tflops": 1951.4, "bf16_tflops_sustained": 1707.8}
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak(peaks, at_max)[0] == 1951.4
    assert bench.tensor_peak(peaks, {})[0] == 1951.4               # no samples: the larger one
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.tensor_peak(peaks, capped)[0] == 1707.8
    slow = {"sm_mhz": 1600.0, "sm_max_mhz": 2070.0, "reasons": []}
    p, label = bench.tensor_peak(peaks, slow)
    assert p == 1707.8 and label.startswith("sustained")



def test_headline_and_further_workloads(bench):
    """The default run puts the largest single-GPU layer in the headline and
    records decode, prefill and replica beside it; any other headline or
    step variant records none unless --also names them."""
    import argparse
    base = dict(workload=bench.HEADLINE, also="auto", gather=False, unpacked=False,
                masked_cap=0, fp8_dispatch=False, replica_relax="", graph=False, zipf=None,
                tokens=0, experts=0)
    ns = lambda **kw: argparse.Namespace(**{**base, **kw})
    assert bench.HEADLINE == "group_limited"
    assert bench.extra_workloads(ns()) == ["decode", "prefill", "replica"]
    assert bench.extra_workloads(ns(workload="prefill")) == []
    assert bench.extra_workloads(ns(gather=True)) == []
    assert bench.extra_workloads(ns(also="none")) == []
    assert bench.extra_workloads(ns(workload="prefill", also="decode,prefill")) == ["decode"]
    rec = {"value": 1.0, "e2e": {}, "cpu_baseline": {}, "stages": {}, "clocks": {}}
    assert set(bench.compact_record(rec)) == {"value", "stages", "clocks"}


def test_traffic_is_scaled_from_the_committed_capture(bench, tmp_path, monkeypatch):
    """roofline.traffic: the capture's DRAM bytes per algorithmic byte times
    the full launch's algorithmic bytes, and nothing once the kernel source
    differs from the captured one."""
    import json
    rec = {"kernel_sha256": bench.kernel_source_hash(),
           "workloads": {"prefill": {"case": "small", "command": "cmd", "dram_bytes_read": 900,
                                     "dram_bytes_write": 110, "algorithmic_bytes": 1000}}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    t, src = bench.measured_traffic("prefill", 5000)
    assert t == 5050 and "1.010 per algorithmic byte" in src
    assert bench.measured_traffic("decode", 5000) == (None, None)
    rec["kernel_sha256"] = "0" * 64
    f.write_text(json.dumps(rec))
    assert bench.measured_traffic("prefill", 5000) == (None, None)
    # the committed record covers every bench workload and matches the sources
    with open(os.path.join(ROOT, "profiles", "grouped_ffn_traffic.json")) as fh:
        committed = json.load(fh)
    assert set(committed["workloads"]) >= {"group_limited", "prefill", "replica", "decode"}
