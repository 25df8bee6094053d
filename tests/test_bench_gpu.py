"""bench.py on the GPU: one short run of the full-size step with the
end-to-end leg, checked for the keys and units of its JSON line (the
timed-region contract: warm-up and step counts, the roofline of the
dominant kernel, clocks, the end-to-end figure and the launch count)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra, steps=5):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(steps), "--warmup", "3",
           "--no-cpu-baseline", *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_json_line_contract():
    d = _run("--legs", "e2e")
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["dtype"] == "bf16" and d["data"].startswith("synthetic")
    cfg = d["config"]
    assert "4096 tokens, hidden 7168, 256 experts / 8 virtual ranks, top-8" in cfg["workload"]
    assert (cfg["T"], cfg["H"], cfg["E"], cfg["R"], cfg["K"]) == (4096, 7168, 256, 8, 8)
    assert "flushed" in cfg["l2"]
    # the step's bytes / time is the value; the value is the layout + dispatch + combine bytes
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["kernel"] == "combine_kernel<8>"
    assert rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert 0.3 < rf["frac"] < 1.5
    assert rf["traffic"] is None or rf["traffic"] > 0.5 * rf["algorithmic_bytes"]
    e2e = d["e2e"]
    assert e2e["unit"] == "GB/s" and 0 < e2e["value"] < d["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 4 * d["steps"]
    clk = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)
    assert e2e["steps"] >= 20
    assert 0.3 < rf["frac_spec"] < rf["frac"]
    assert rf["pair"]["bytes"] == d["ops"]["dispatch_bf16"]["bytes"] + rf["algorithmic_bytes"]
    assert 0.3 < rf["pair"]["frac"] < 1.5 and 0.3 < rf["combine_alone"]["frac"] < 1.5
    assert rf["traffic"] is None or rf["traffic_source"].startswith("profiles/")
    ops = d["ops"]
    for key in ("layout", "dispatch_bf16", "combine"):
        assert ops[key]["us"] > 0 and ops[key]["eager_us"] > 0
    for key in ("dispatch_bf16", "combine", "dispatch_combine_pair"):
        assert ops[key]["bytes"] > 0 and 0.2 < ops[key]["frac"] < 1.5


def test_bench_other_workload_as_the_step():
    d = _run("--legs", "none", "--workload", "ds16_wide")
    cfg = d["config"]
    assert (cfg["T"], cfg["H"], cfg["E"], cfg["R"], cfg["K"]) == (16384, 2048, 64, 32, 6)
    assert "32 ranks" in cfg["workload"] and d["roofline"]["kernel"] == "combine_kernel<6>"
    assert d["value"] > 0 and "e2e" not in d
    assert d["roofline"]["traffic"] is None            # the committed capture is of the DeepSeek-V3 shape


def test_bench_fp8_step_and_format_legs():
    """--workload dsv3_fp8 times layout -> FP8 dispatch -> combine as the
    step; the format leg adds the bf16 step and the FP8 / MXFP8 dispatches."""
    d = _run("--legs", "formats", "--workload", "dsv3_fp8")
    assert d["dtype"] == "e4m3+bf16" and d["config"]["step"].startswith("layout + FP8")
    ops = d["ops"]
    assert ops["dispatch_fp8"]["bytes"] == 218_836_384 and ops["dispatch_mxfp8"]["bytes"] == 218_836_384
    assert ops["step_bf16"]["us"] > ops["dispatch_combine_pair"]["us"] > 0
    for key in ("dispatch_fp8", "dispatch_mxfp8"):
        assert 0.3 < ops[key]["frac"] < 1.5 and ops[key]["eager_us"] > 0
    # the step's bytes: layout + FP8 dispatch + combine
    step_bytes = ops["layout"]["bytes"] + 218_836_384 + d["roofline"]["algorithmic_bytes"]
    assert abs(d["value"] * 1e9 * d["ms_per_step"] * 1e-3 / step_bytes - 1) < 1e-3


def test_bench_fewer_steps_than_buffer_placements():
    """The timed steps rotate over four buffer placements; three steps
    (the launch-list profile's command) report the three placements timed."""
    d = _run("--legs", "none", steps=3)
    assert d["steps"] == 3 and d["value"] > 0
    assert len(d["ops"]["step_us_by_placement"]) == 3
