"""The benchmark's JSON line on a GPU: one line with the metric, the whole-job
value, the roofline of the dominant kernel against the measured peak, the
CPU baseline (the oracle), the end-to-end figure with its copied bytes,
sampled clocks and the count of this library's kernel launches."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keys_on_a_small_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny",
                          "--steps", "5", "--warmup", "3", "--e2e-steps", "3",
                          "--workload-steps", "5"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"].startswith("tiny: W=2 logical ranks")
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert c["single_thread"]["cores"] == 1 and c["single_thread"]["value"] > 0
    assert d["oracle_parity"].startswith("bit-exact")
    e = d["e2e"]
    assert e["value"] > 0 and e["output_check"] == "pass"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * 5          # tiny: copy (with the layout) + combine
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["identity_check"] == "pass" and d["device_errors"] == 0
    # every workload of the benchmark, measured in the same run
    wls = d["workloads"]
    assert list(wls) == ["tiny", "dsv3", "dsv3_fp8_zipf", "ll_decode", "mixtral"]
    for name, e in wls.items():
        assert e["ms_per_step"] > 0 and e["tokens_per_s"] > 0 and e["gb_per_s"] > 0, name
        assert 0 < e["frac_of_measured_hbm"] and 0 < e["dominant_frac_of_measured_hbm"], name
        assert e["identity_check"] == "pass", name
        assert e["oracle_parity"].startswith("bit-exact"), name
        assert e["cpu_baseline"]["kind"] == "oracle" and e["cpu_baseline"]["value"] > 0, name
    assert wls["ll_decode"]["mode"].startswith("split phases")
    assert wls["tiny"]["cold_l2_ms_per_step"] > 0 and wls["ll_decode"]["cold_l2_ms_per_step"] > 0
