"""The benchmark's host-side pieces, without a GPU: the reference arm's JSON
line, the clock-sample parsing and the traffic lookup."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1", "--n", "1048576"],
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["metric"] == bench.METRIC


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--n", "65536"],
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_sampler_parses_and_flags_reasons():
    cs = bench.ClockSampler(0)
    cs.proc = object()  # pretend the sampler ran

    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    cs.proc = _P()
    cs.t_start, cs.t_stop = 100.0, 101.0
    cs.lines = [
        (99.0, "0, 1000, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (100.2, "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (100.5, "0, 2040, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (100.8, "0, 2070, 2070, 1250.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
    ]
    out = cs.stop()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3
    assert out["window"] == "timed region"


def test_traffic_lookup_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    from memory_bound_elementwise_gb300 import _build
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = {"add_f32_v256": {"dram_bytes_per_launch": 123, "source_digest": _build.source_digest(),
                             "note": "x"}}
    (prof / "traffic.json").write_text(json.dumps(good))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("add_f32_v256")[0] == 123
    good["add_f32_v256"]["source_digest"] = "0" * 64
    (prof / "traffic.json").write_text(json.dumps(good))
    assert bench.profiled_traffic("add_f32_v256")[0] is None
    assert bench.profiled_traffic("missing")[0] is None
