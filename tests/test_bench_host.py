"""Host-side pieces of bench.py that need no GPU: workload selection (dtype
override, sub-batch), the config record of each option, and the traffic
record that is reported only for the kernel source it was measured on."""
import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from rnn_transducer_loss_gb300 import workloads as W  # noqa: E402


def _args(**kw):
    a = dict(workload="tiny", dtype=None, samples=0, gpus=1, padded=False, fastemit=0.0,
             big_blanks="", sigma=0.0)
    a.update(kw)
    return argparse.Namespace(**a)


def test_dtype_override_keeps_the_values_distribution():
    base = bench.make_workload(_args(), "cpu")
    bf = bench.make_workload(_args(dtype="bf16"), "cpu")
    assert bf.logits.dtype == torch.bfloat16 and bf.cfg.name == "tiny_bf16"
    # same seeded draws, rounded to the other storage type
    torch.testing.assert_close(bf.logits.float(), base.logits.to(torch.bfloat16).float())
    np.testing.assert_array_equal(bf.T, base.T)
    np.testing.assert_array_equal(bf.targets, base.targets)


def test_subset_keeps_the_first_samples():
    full = bench.make_workload(_args(workload="char_asr"), "cpu")
    sub = bench.make_workload(_args(workload="char_asr", samples=5), "cpu")
    assert sub.cfg.B == 5 and sub.rows == int(full.offsets[5])
    assert torch.equal(sub.logits, full.logits[:sub.rows])


def test_config_records_options():
    wl = bench.make_workload(_args(), "cpu")
    plain = bench.config_of(wl, _args(), l2="flushed")
    assert plain["workload"] == "tiny" and plain["l2"] == "flushed"
    assert "layout" not in plain and "fastemit_lambda" not in plain
    cfg = bench.config_of(wl, _args(padded=True, fastemit=0.01, big_blanks="2,4", sigma=0.05),
                          l2="flushed")
    assert cfg["layout"].startswith("padded (B, max_T, max_U+1, V) = (2, 8, 4, 16)")
    assert cfg["fastemit_lambda"] == 0.01
    assert cfg["big_blank_durations"] == [2, 4] and cfg["sigma"] == 0.05


def test_padded_layout_of_a_workload():
    wl = W.make("tiny", "cpu")
    xp = W.to_padded(wl, fill=float("nan"))
    assert xp.shape == (2, 8, 4, 16)
    for b in range(2):
        T, U = int(wl.T[b]), int(wl.U[b])
        assert torch.equal(xp[b, :T, :U + 1].reshape(-1, 16), wl.logits[wl.sample_rows(b)])
        assert torch.isnan(xp[b, T:]).all() and torch.isnan(xp[b, :, U + 1:]).all()


def test_traffic_record_matches_only_its_source(tmp_path, monkeypatch):
    v = bench.recorded_traffic("persistent_main", "bpe_asr")
    # a record is reported only for the kernel source it was taken on
    assert v is None or v > 1.9e9
    assert bench.recorded_traffic("persistent_main", "char_asr") is None
    stale = tmp_path / "traffic.txt"
    stale.write_text("source_sha256_16=0000000000000000\nworkload=bpe_asr\n"
                     "persistent_main.dram_bytes_per_launch=123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(stale))
    assert bench.recorded_traffic("persistent_main", "bpe_asr") is None
    fresh = tmp_path / "fresh.txt"
    fresh.write_text(f"source_sha256_16={bench.kernel_source_hash()}\nworkload=bpe_asr\n"
                     "persistent_main.dram_bytes_per_launch=123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(fresh))
    assert bench.recorded_traffic("persistent_main", "bpe_asr") == 123.0
    assert bench.recorded_traffic("no_such_kernel", "bpe_asr") is None


def test_peak_is_measured_or_the_stated_fallback():
    peak, kind = bench.load_peak()
    assert kind in ("measured", "fallback")
    assert (peak == bench.FALLBACK_HBM_GBS) == (kind == "fallback")


def test_clock_lines_parse_and_window_filter():
    import datetime as dt
    lines = [
        "2026/12/02 15:49:01.000, 0, 1200, 2070, 150.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 15:49:01.020, 0, 2070, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 15:49:01.040, 0, 2055, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "2026/12/02 15:49:01.200, 0, 1100, 2070, 120.0, 0x0, Not Active, Active, Not Active, Not Active",
    ]
    samples = bench.parse_clock_lines(lines)
    assert len(samples) == 4
    t = lambda ms: dt.datetime(2026, 12, 2, 15, 49, 1, ms * 1000)   # noqa: E731
    inside = bench.summarize_clocks(samples, t(10), t(50))
    assert inside["samples"] == 2 and inside["sm_mhz"] == (2070 + 2055) / 2
    assert inside["reasons"] == ["sw_power_cap"] and "note" not in inside
    # a window shorter than the sampling period: the nearest samples, said so
    near = bench.summarize_clocks(samples, t(21), t(23))
    assert near["samples"] == 3 and "note" in near
    assert bench.summarize_clocks([], t(0), t(1))["reasons"] == ["no samples"]


def test_clock_lines_without_readable_timestamps_use_all_samples():
    import datetime as dt
    lines = ["Tue Dec  2 15:49:01 2026, 0, 2070, 2070, 900, 0x0, Not Active, Not Active, "
             "Not Active, Not Active"] * 3
    samples = bench.parse_clock_lines(lines)
    assert len(samples) == 3 and samples[0][0] is None
    now = dt.datetime.now()
    out = bench.summarize_clocks(samples, now, now)
    assert out["samples"] == 3 and out["sm_mhz"] == 2070 and "note" in out


def test_roofline_uses_the_kernel_time_and_refuses_a_kernel_longer_than_the_step():
    r = bench.kernel_roofline("persistent_main", 1.969e9, 0.4, 0.4, 6786.9, "measured", None)
    assert abs(r["frac"] - 1.969e9 / 0.4e-3 / 1e9 / 6786.9) < 1e-12
    # One outlier stage sample (2.83 ms against a 0.40 ms step) is refused.
    r = bench.kernel_roofline("persistent_main", 1.969e9, 2.83, 0.40, 6786.9, "measured", None)
    assert r["frac"] is None and r["achieved"] is None and "exceeds" in r["note"]


def test_algorithmic_bytes_fused_and_not():
    # fused: one read of every logit + one write of every gradient element
    assert bench.algorithmic_bytes(True, 1000, 10, 1000, 2) == 4000
    # not fused: the gradient write + the blank and label gathers of each row
    assert bench.algorithmic_bytes(False, 811040 * 512, 811040, 811040 * 512, 2) == \
        811040 * 512 * 2 + 2 * 2 * 811040


def test_clock_summary_counts_the_timed_samples_inside_a_loaded_window():
    import datetime as dt
    t = dt.datetime(2026, 1, 1)
    ms = lambda k: t + dt.timedelta(milliseconds=k)   # noqa: E731
    samples = [(ms(k), 2070.0 - (k == 500), 2070.0, set()) for k in range(0, 700, 20)]
    out = bench.summarize_clocks(samples, ms(600), ms(640), loaded_begin=ms(100))
    assert out["samples"] == sum(1 for k in range(0, 700, 20) if 100 <= k <= 640)
    assert out["samples_timed"] == 3 and out["sm_mhz"] == 2070.0 and out["reasons"] == []
    out = bench.summarize_clocks(samples, ms(600), ms(640))
    assert out["samples"] == 3


def test_dp_latency_from_a_trace():
    T = np.array([10, 20], dtype=np.int32)
    U = np.array([5, 0], dtype=np.int32)
    rec = {"kind": np.array([0, 1, 1]), "sample": np.array([0, 0, 1]),
           "sm": np.array([0, 1, 2]), "start_us": np.array([0.0, 1.0, 2.0]),
           "end_us": np.array([1.0, 4.0, 6.0])}
    d = bench.dp_latency(rec, T, U)
    assert d["samples"] == 2
    assert abs(d["max_ns"] - 3000 / 15) < 1e-9 and abs(d["min_ns"] - 4000 / 20) < 1e-9
    assert d["longest_lattice"]["T"] == 20
