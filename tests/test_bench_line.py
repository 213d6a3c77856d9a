"""The bench's JSON line, built on the CPU from made-up timings: `steps` is
the K the command asked for (the per-chunk breakdown sits under its own
key), the prefill roofline divides by the burst peak for a timed region
under a second and by the sustained one otherwise, and the per-launch DRAM
traffic of a committed ncu summary is reported only while the recorded
source hash matches the current prefill sources."""
import os

import bench


def _r(total_ms, K=20):
    chunks = [{"chunk": c, "rows": 2048, "context": 2048 * (c + 1), "step_us": 500.0,
               "append_us": 9.0, "prefill_us": 300.0, "prefill_TFLOPs": 1000.0,
               "decode_us": 190.0, "decode_GBps": 5000.0} for c in range(14)]
    return dict(total_ms=total_ms, step_ms=0.5, balanced=True, app_ms=0.009 * K,
                pre_ms=0.3 * K, dec_ms=0.19 * K, flops=3.0e11 * K, dbytes=1.0e9 * K,
                launches=4 * K, clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
                chunks=chunks)


PEAKS = (6686.8, 1953.3, 1742.8, "measured", 1477.0)


def test_steps_is_the_requested_count():
    line = bench.make_line(20, 5, 1, _r(10.0), (520.0, 1, 2, 28), PEAKS, {}, {"workload": "x"})
    assert line["steps"] == 20 and line["warmup"] == 5
    assert isinstance(line["chunk_steps"], list) and len(line["chunk_steps"]) == 14
    assert line["value"] == 500.0 and line["e2e"]["steps"] == 28


def test_frac_uses_the_burst_peak_for_a_short_region_and_sustained_for_a_long_one():
    short = bench.make_line(20, 5, 1, _r(10.0), (1, 1, 1, 28), PEAKS, {}, {})["roofline"]
    assert short["peak"] == 1953.3
    assert abs(short["frac"] - 1000.0 / 1953.3) < 1e-4
    long_ = bench.make_line(20, 5, 1, _r(2000.0), (1, 1, 1, 28), PEAKS, {}, {})["roofline"]
    assert long_["peak"] == 1742.8
    assert short["frac_of_spec_dense_bf16"] == round(1000.0 / 2250.0, 4)
    assert abs(short["frac_clock_normalized"] - 1000.0 / (1953.3 * 2070.0 / 1477.0)) < 1e-4


def test_overlapped_schedule_reports_the_prefill_sm_share():
    r = _r(10.0)
    r.update(overlap=True, sm_share=0.75)
    line = bench.make_line(20, 5, 1, r, (1, 1, 1, 28), PEAKS, {}, {})
    roof = line["roofline"]
    assert roof["peak"] == 1953.3                      # the measured peak itself
    assert abs(roof["frac"] - 1000.0 / 1953.3) < 1e-4
    assert roof["sm_share"] == 0.75
    assert abs(roof["frac_of_sm_share"] - 1000.0 / 1953.3 / 0.75) < 1e-4
    assert line["schedule"].startswith("overlapped")
    seq = bench.make_line(20, 5, 1, _r(10.0), (1, 1, 1, 28), PEAKS, {}, {})
    assert "sm_share" not in seq["roofline"] and seq["schedule"].startswith("sequential")
    assert "sequential" not in seq
    # with the same steps timed one after the other as well
    alone = _r(10.0, K=280)
    alone.update(steps=280, pre_ms=0.28 * 280, flops=4.0e11 * 280, dec_ms=0.2 * 280,
                 dbytes=1.3e9 * 280)
    r.update(alone=alone)
    line = bench.make_line(20, 5, 1, r, (1, 1, 1, 28), PEAKS, {}, {})
    a_tf = 4.0e11 / 0.28e-3 / 1e12
    assert abs(line["roofline"]["achieved_alone"] - round(a_tf, 1)) < 1e-6
    assert abs(line["sequential"]["prefill"]["frac_of_measured_burst"] - a_tf / 1953.3) < 1e-4
    assert abs(line["sequential"]["decode"]["GBps"] - 1.3e9 / 0.2e-3 / 1e9) < 1e-6
    assert line["sequential"]["steps"] == 280


def test_traffic_only_from_a_capture_of_the_current_sources(tmp_path, monkeypatch):
    cur = bench.sources_sha256(bench.PREFILL_SOURCES)
    f = tmp_path / "prof.md"
    f.write_text(f"dram_bytes_per_launch_mixed_step = 1.25e8  (sha256 {cur})\n"
                 f"tensor_pipe_active_pct_2048x16384 = 61.5  (sha256 {'0' * 64})\n")
    monkeypatch.setattr(bench, "PREFILL_PROFILE", str(f))
    prof = bench.prefill_profile()
    assert prof == {"dram_bytes_per_launch_mixed_step": 1.25e8}
    roof = bench.make_line(20, 5, 1, _r(10.0), (1, 1, 1, 28), PEAKS, prof, {})["roofline"]
    assert roof["traffic"] == 1.25e8 and "ncu_tensor_pipe_active_pct" not in roof
    monkeypatch.setattr(bench, "PREFILL_PROFILE", os.path.join(str(tmp_path), "missing.md"))
    assert bench.prefill_profile() == {}
