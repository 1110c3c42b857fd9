"""Host logic of bench.py that runs without a GPU: the clock-record parser, the
step-time distribution, the oracle sampler of the CPU baseline and the JSON
line of the reference arm."""
import json
import os

import numpy as np
import pytest

import bench
import workloads as W


class _Done:
    """Stands in for a finished nvidia-smi process."""


def _sampler_with(lines, tmp_path):
    s = bench.ClockSampler(0)
    f = open(tmp_path / "clocks.csv", "w+")
    f.write("\n".join(lines) + "\n")
    s.f, s.proc = f, _Done()
    return s


def test_clock_summary_median_max_and_reasons(tmp_path):
    row = "0, {sm}, 2070, 900.1, 0x0, {hw}, Not Active, Not Active, {cap}"
    lines = [row.format(sm=sm, hw="Not Active", cap="Not Active") for sm in (2070, 2055, 2070)]
    lines.append(row.format(sm=1980, hw="Not Active", cap="Active"))
    lines.append("garbage line")
    d = _sampler_with(lines, tmp_path).summary()
    assert d["sm_mhz"] == 2062.5 and d["sm_max_mhz"] == 2070.0 and d["samples"] == 4
    assert d["reasons"] == ["sw_power_cap"]
    lines.append(row.format(sm=1500, hw="Active", cap="Not Active"))
    d = _sampler_with(lines, tmp_path).summary()
    assert d["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_nvidia_smi():
    d = bench.ClockSampler(0).summary()
    assert d["sm_mhz"] is None and d["reasons"] == ["nvidia-smi unavailable"]


def test_step_distribution():
    assert bench.step_distribution([]) is None
    d = bench.step_distribution([1.0] * 9 + [2.0])               # ms
    assert d["median"] == 1000.0 and d["p10"] == 1000.0 and d["steps"] == 10
    assert d["p90"] == pytest.approx(1100.0)


def test_peak_is_the_measured_copy_bandwidth():
    gbs, kind = bench.peaks()
    p = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        assert kind == "measured" and gbs == float(json.load(open(p))["hbm_gbs"])
    else:
        assert kind == "fallback" and gbs == 6800.0


def test_oracle_sample_scales_by_tokens():
    b = W.make_batch([300, 50, 700], Hq=16, Hkv=2, seed=3)
    per_batch, threads, desc = bench.oracle_sample(b, 0.05)
    assert per_batch > 0 and threads == (os.cpu_count() or 1)
    assert "of 3 requests" in desc and "of 1050 tokens" in desc


def test_reference_line_contract(monkeypatch):
    monkeypatch.setattr(bench, "oracle_sample", lambda b, s: (0.25, 7, "fake sample"))

    class A:
        config, seed, warmup, steps, requests = 1, 0, 3, 2, None

    line = bench.run_reference(A, rank=0, world=1)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == bench.UNIT and line["higher_is_better"] is False
    assert line["value"] == 250000.0 and line["ms_per_step"] == 250.0
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == W.CONFIGS[1] and line["config"]["batch"] == 3
    assert line["cpu_baseline"] == {"value": 250000.0, "unit": bench.UNIT, "cores": 7,
                                    "kind": "oracle", "sample": "fake sample"}
    assert line["e2e"] == {"value": 250000.0, "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    json.dumps(line)                                           # one JSON line


@pytest.mark.parametrize("rows,attn,expect", [
    (8, "auto", 1), (16, "auto", 1), (16, "mma", 1), (16, "tc", None),
    (32, "auto", 1), (32, "tc", 1), (32, "mma", None), (64, "auto", 1),
    (48, "allheads", 3), (8, "allheads", 1)])
def test_traced_tail_follows_the_timed_kernel(rows, attn, expect):
    """The tail is traced only when the traced call runs the kernel the bench times: the
    tcgen05 kernel above 16 rows per KV head (one trace row per CTA), mma.sync up to 16
    (one per row group), the all-heads variant always."""
    assert bench.traced_groups(rows, attn) == expect
