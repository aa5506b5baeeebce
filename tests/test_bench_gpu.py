"""bench.py end to end on the GPU: the headline line is the last line of
stdout, parses, stays compact, and carries the checked parity, roofline,
cpu_baseline, e2e and clock records."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_headline_is_the_last_line_and_checked():
    n = 1 << 24
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
                        "--n", str(n), "--no-aux"], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 2
    aux, head = json.loads(lines[0]), json.loads(lines[-1])
    assert aux["aux_of"] == head["metric"]
    assert len(lines[-1].encode()) < 4096
    assert head["parity"] == "bit-exact vs the CPU oracle"
    assert head["value"] > 0 and head["steps"] == 5 and head["warmup"] == 3 and head["gpu_launches"] == 5
    assert head["config"]["n"] == n
    roof = head["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    cpu = head["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0 and cpu["unit"] == "GB/s"
    e2e = head["e2e"]
    assert e2e["h2d_bytes_per_step"] == 8 * n and e2e["d2h_bytes_per_step"] == 4 * n
    assert e2e["value"] > 0 and e2e["result_matches_device"] is True
    link = e2e["link"]
    assert 0 < link["h2d_gbps"] and 0 < link["d2h_gbps"] and 0 < link["both_gbps"]
    assert e2e["frac_of_link_both"] == pytest.approx(e2e["value"] / link["both_gbps"])
    assert head["clocks"]["sm_mhz"] is None or head["clocks"]["sm_mhz"] > 0
