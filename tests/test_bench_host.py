"""Host-side logic of bench.py that needs no GPU: the clock-sample summary
(median SM clock and the throttle reasons seen) and the gate that reports the
committed ncu traffic only while the decode sources are the profiled ones."""
import os

import bench


def _sampler(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(l + "\n" for l in lines))
    s = bench.ClockSampler(0)
    s.path = str(path)
    s.proc = object()          # a sampler that ran
    return s


def test_clock_summary_median_and_reasons(tmp_path):
    rows = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1300.1, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    got = _sampler(tmp_path, rows).summary()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_reports_thermal_and_hw_slowdown(tmp_path):
    rows = ["0, 1500, 2070, 1390, 0x48, Active, Not Active, Active, Not Active"]
    got = _sampler(tmp_path, rows).summary()
    assert got["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and got["sm_mhz"] == 1500.0


def test_clock_summary_without_samples(tmp_path):
    assert _sampler(tmp_path, []).summary() is None
    s = bench.ClockSampler(0)
    s.proc = None              # nvidia-smi could not be started
    assert s.summary() is None


def test_decode_source_hash_ignores_comments_only():
    # a comment edit leaves the kernel (and the profiled traffic) valid; a code edit does not
    a = "int f(int x) {  // twice\n    /* doubled\n       here */ return 2 * x;\n}\n"
    b = "int f(int x) {\n\n    return 2 * x;   \n}\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_profiled_traffic_follows_the_decode_sources(tmp_path, monkeypatch):
    # the traffic is reported only while the summary carries the hash of the current decode sources
    fake = tmp_path / "profile.txt"
    fake.write_text("decode_source_sha256: 0000000000000000\ntraffic_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(fake))
    assert bench._profiled_traffic() is None            # stale: another source version
    fake.write_text(f"decode_source_sha256: {bench._decode_source_sha()}\ntraffic_bytes_per_launch: 123\n")
    assert bench._profiled_traffic() == 123
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.txt"))
    assert bench._profiled_traffic() is None


def test_peaks_come_from_the_measured_file_when_present():
    peak, kind = bench._peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and peak > 1000
    else:
        assert kind == "fallback"


def test_bucket_report_follows_the_oracle_and_the_page_formula():
    """config4_bytes: needed_seq and the bucket as the oracle's decode_bucket gives them ("Decode
    Context-Length Bucketing", Design / Per-step bucket selection), bytes at token granularity."""
    import numpy as np

    import oracle
    from paged_kv_cache_slot_gb300 import workloads as wl

    w = wl.make("long_context")
    rep = bench.bucket_report(w)
    mml = w.extra["max_model_len"]
    want = oracle.decode_bucket(w.prior_lens, w.q_len - 1, w.extra["buckets"], mml)
    assert rep["bucket"] == want
    assert rep["needed_seq"] == int(w.prior_lens.max()) + 1 + (w.q_len - 1)
    per_tok = 2 * w.num_kv_heads * w.head_dim * 2
    assert rep["kv_bytes_read"] == int(w.context_lens.astype(np.int64).sum()) * per_tok
    assert rep["full_row_bytes"] == 8 * 131072 * 4096
    assert rep["bucketed_bytes"] == 8 * want * 4096
    # a batch whose longest request needs more than the largest bucket falls back to max_model_len
    w.prior_lens = np.array([100, 20000, 5, 7, 9, 11, 13, 15], np.int64)
    rep = bench.bucket_report(w)
    assert rep["bucket"] == oracle.decode_bucket(w.prior_lens, 0, w.extra["buckets"], mml) == mml
    assert rep["full_row_over_read"] > rep["bucketed_over_read"] - 1e-12
