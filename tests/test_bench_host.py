"""Host logic of bench.py (no GPU): the algorithmic byte counts behind the roofline, and the rule
that a committed DRAM-traffic figure is reported only while the kernel's sources are unchanged."""
import json
import os
import sys
import types

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _wl(fmt, T, H, I, E, ids):
    return types.SimpleNamespace(fmt=fmt, T=T, H=H, I=I, E=E, topk=8, ids=torch.tensor(ids, dtype=torch.int32))


def test_matrix_bytes_fp8_and_nvfp4():
    # FP8: one byte per code + one fp32 per 128x128 block; NVFP4: half a byte per code + one byte per 16
    assert bench.matrix_bytes("fp8", 2048, 7168) == 2048 * 7168 + 16 * 56 * 4
    assert bench.matrix_bytes("nvfp4", 1536, 5120) == 1536 * 5120 // 2 + 1536 * 320


def test_alg_bytes_counts_each_distinct_expert_once():
    H, I = 7168, 2048
    # two tokens sharing expert 3; -1 and an out-of-range id add nothing
    ids = [[3, 1, 2, 4, 5, 6, 7, 8], [3, 9, 10, 11, 12, -1, 99, 13]]
    b = bench.alg_bytes(_wl("fp8", 2, H, I, 16, ids))
    distinct = 13   # {1..13} minus nothing: 3 counted once, -1 and 99 dropped
    assert b["distinct"] == distinct
    w = distinct * (2 * bench.matrix_bytes("fp8", I, H) + bench.matrix_bytes("fp8", H, I))
    assert b["weights"] == w
    assert b["total"] == w + 2 * H * 2 + 2 * H * 2 + 16 * 8
    # the single-token decode figure quoted in the docs: 8 experts x 3 x 7168 x 2048 codes + scales
    one = bench.alg_bytes(_wl("fp8", 1, H, I, 256, [list(range(8))]))
    assert one["weights"] == 8 * 3 * (H * I + 16 * 56 * 4)


def test_profiled_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "moe_expert_ffn_histogram_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (csrc / "h.cuh").write_text("header v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha(["k.cu", "h.cuh"])
    entry = {"files": ["k.cu", "h.cuh"], "source_sha": sha, "dram_bytes_per_launch": 1234}
    (prof / "traffic.json").write_text(json.dumps({"cfg": {"kern": entry}}))
    assert bench.profiled_traffic("cfg", "kern") == 1234
    assert bench.profiled_traffic("cfg", "other") is None
    assert bench.profiled_traffic("nope", "kern") is None
    (csrc / "h.cuh").write_text("header v2")               # the kernel changed since the capture
    assert bench.profiled_traffic("cfg", "kern") is None
    # a file outside the list does not matter
    (csrc / "h.cuh").write_text("header v1")
    (csrc / "unrelated.cu").write_text("x")
    assert bench.profiled_traffic("cfg", "kern") == 1234


def test_committed_traffic_entries_are_well_formed():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for cfg, kernels in d.items():
        if cfg.startswith("_"):
            continue
        for name, e in kernels.items():
            assert e["dram_bytes_per_launch"] == e["read"] + e["write"], (cfg, name)
            assert e["files"] and all(os.path.exists(os.path.join(ROOT, "moe_expert_ffn_histogram_gb300",
                                                                  "csrc", f)) for f in e["files"]), (cfg, name)


def test_cpu_baseline_fills_its_budget():
    # every seeded route set is run until its share of the budget is used
    cb = bench.cpu_baseline("tiny_fp8_decode", torch.device("cpu"), budget_s=0.8)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["cores"] >= 1
    secs = float(cb["sample"].split(", ")[-1].split()[-2])
    assert 0.4 <= secs <= 1.6, cb["sample"]
    toks = int(cb["sample"].split()[0])
    assert toks >= bench.N_ROUTE_SETS
    assert abs(cb["value"] - toks / secs) / cb["value"] < 0.1


def test_nearest_rank_on_the_gate_binary_example():
    # "memra-engine 0.108.0 src/bin/ep_step_fp8_gate.rs", test nearest_rank_percentiles_use_observed_samples
    samples = [10, 20, 30, 40, 50]
    assert bench.nearest_rank(samples, 50) == 30
    assert bench.nearest_rank(samples, 90) == 50
    assert bench.nearest_rank(samples, 95) == 50
    assert bench.nearest_rank(samples, 99) == 50
    assert bench.nearest_rank(samples, 1) == 10 and bench.nearest_rank(samples, 100) == 50
    st = bench.step_stats_us([0.001 * v for v in (5, 1, 4, 2, 3)])
    assert st["min"] == 1.0 and st["max"] == 5.0 and st["p50"] == 3.0 and st["mean"] == 3.0


def _fold(values):
    s = 0x9E3779B97F4A7C15
    for v in np.asarray(values, dtype=np.float32).view(np.uint32):
        s = (((s << 7) | (s >> 57)) & 0xFFFFFFFFFFFFFFFF) ^ int(v)
    return s


def test_output_checksum_matches_the_sequential_fold_and_is_bit_sensitive():
    # the gate binary's test output_checksum_is_bit_sensitive_and_repeat_stable
    vals = [0.0, -0.0, 1.0, -2.5]
    assert bench.output_checksum(vals) == bench.output_checksum(vals)
    assert bench.output_checksum(vals) != bench.output_checksum([0.0, 0.0, 1.0, -2.5])
    # the closed form equals the fold taken one value at a time (lengths across the 64-bit period)
    rng = np.random.default_rng(3)
    for n in (0, 1, 2, 9, 10, 63, 64, 65, 1000):
        v = rng.standard_normal(n).astype(np.float32)
        assert bench.output_checksum(v) == _fold(v), n


def test_graded_fraction_takes_the_larger_floor():
    # 6.7734 GB at 6,773.4 GB/s is 1 ms; 1.93 TFLOP at 1,930 TFLOP/s is 1 ms; a 2 ms step is 0.5
    f, floor = bench.graded_fraction(6.7734e9, 1.93e12, 2e-3, 6773.4, 1930.0)
    assert abs(floor - 1e-3) < 1e-9 and abs(f - 0.5) < 1e-9
    f, floor = bench.graded_fraction(13.5468e9, 1.93e12, 4e-3, 6773.4, 1930.0)   # bytes dominate
    assert abs(floor - 2e-3) < 1e-9 and abs(f - 0.5) < 1e-9


def test_sweep_rows_even_split():
    """The narrow tiers' split of T tokens into ceil(T/8) even sweeps, never a trailing sweep of
    one (forward.rs, `moe_row_groups`), as bench.py models it."""
    assert bench.sweep_rows(9) == [5, 4]
    assert bench.sweep_rows(16) == [8, 8]
    assert bench.sweep_rows(17) == [6, 6, 5]
    for T in range(1, 300):
        r = bench.sweep_rows(T)
        assert sum(r) == T and len(r) == (T + 7) // 8 and max(r) - min(r) <= 1 and max(r) <= 8


def test_ceiling_entry_ratio_and_fraction():
    """The size-matched read ceiling: bytes / read time against the peak, and the read time over
    the measured time (1.0 = the kernel or step ran as fast as a plain read of its bytes)."""
    e = bench.ceiling_entry(352_436_288, 72.3, 61.44, 6773.5, "step_vs_read")
    assert e["bytes"] == 352_436_288
    assert e["read_gbs"] == pytest.approx(352_436_288 / 61.44e-6 / 1e9, rel=1e-3)
    assert e["read_frac_of_peak"] == pytest.approx(352_436_288 / 61.44e-6 / 1e9 / 6773.5, abs=1e-4)
    assert e["step_vs_read"] == pytest.approx(61.44 / 72.3, abs=1e-4)
    # a step slower than the read reports a ratio below 1
    assert bench.ceiling_entry(1 << 20, 10.0, 5.0, 1000.0, "kernel_vs_read")["kernel_vs_read"] == 0.5
