"""bench.py's host-side contract on CPU: the reference arm's JSON line (the
oracle timed on a bounded sample), the refusal of fewer than three warm-up
steps, the clock-record summary that decides whether a run is kept, and the
per-workload traffic lookup."""
import json
import math

import pytest

import bench
from bit_quantized_kv_kvq_gb300 import workloads as W

TINY = "tiny-q8_0-gqa8x2-d128-s4096"


def test_reference_arm_prints_one_contract_line(capsys):
    assert bench.main(["--impl", "reference", "--workload", TINY, "--steps", "2", "--warmup", "3"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["value"] > 0 and math.isfinite(d["value"]) and d["ms_per_step"] > 0
    assert d["config"]["workload"] == TINY
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_fewer_than_three_warmup_steps_are_refused():
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--workload", TINY, "--steps", "1", "--warmup", "2"])


def _row(sm, power, hw="Not Active", sw_power="Not Active"):
    return "GPU-abc, %s, 2070, %s, 0x0, %s, Not Active, Not Active, %s\n" % (sm, power, hw, sw_power)


def test_clock_summary_takes_the_loaded_samples_and_lists_reasons(tmp_path):
    p = tmp_path / "clocks.csv"
    # idle samples (low power) are left out of the median under load
    p.write_text(_row(345, 90) + _row(2070, 900) + _row(2055, 950, sw_power="Active") +
                 _row(2070, 910, hw="Active") + _row(600, 100))
    cs = bench.ClockSampler("GPU-abc")
    cs.path = str(p)
    s = cs.summary()
    assert s["gpu"] == "GPU-abc" and s["samples"] == 5
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert not p.exists()


def test_clock_summary_without_samples_says_so(tmp_path):
    p = tmp_path / "empty.csv"
    p.write_text("")
    cs = bench.ClockSampler("GPU-abc")
    cs.path = str(p)
    s = cs.summary()
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"] and s["sm_mhz"] is None


def test_traffic_lookup_by_workload_and_kernel():
    assert bench.load_traffic(W.LLAMA8B_FULL, "decode_attention") == 221622528
    assert bench.load_traffic(W.LLAMA8B_FULL, "prefill") is None
    assert bench.load_traffic(W.BY_NAME[TINY], "decode_attention") is None


def test_gbs_is_bytes_over_milliseconds():
    assert bench.gbs(6.0e9, 1000.0) == pytest.approx(6.0)
    assert bench.gbs(218155040, 0.0629) == pytest.approx(3468.3, rel=1e-4)
