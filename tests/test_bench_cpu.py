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


def _headline(parity=True, note_len=200):
    per = [0.000449, 0.000448, 0.000450]
    return bench.headline_line(
        value=7137.7, parity=parity, world=1, steps=20, warmup=5, total_s=0.009, n=1 << 28, lo=0,
        hi=1 << 28, step_bytes=12 << 28,
        rec={"path": "v256", "vec_bytes": 32, "grid": 65536, "block": 256},
        facts={"sms": 152, "l2_bytes": 135528448, "driver": "580.178.04"}, gpu_name="NVIDIA GB300",
        achieved=7175.7, peak=6796.2, peak_src="measured hbm_gbs (copy, read+write bytes)",
        traffic=3225885696, traffic_note="x" * note_len, kern_s=0.000449, per_launch=sorted(per),
        e2e={"value": 301.4, "unit": "GB/s", "h2d_bytes_per_step": 8 << 28, "d2h_bytes_per_step": 4 << 28,
             "steps": 10, "result_matches_device": True, "how": "y" * 150},
        clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "sm_mhz_min": 2070.0, "reasons": ["sw_power_cap"],
                "samples": 17, "window": "timed region", "source": "NVML"},
        cpu_baseline={"value": 21.0, "unit": "GB/s", "cores": 1, "kind": "oracle",
                      "sample": "3 full passes over the N=2^28 inputs (11.2 s)", "cpu": "aarch64 Neoverse-V2",
                      "all_cores_value": 135.0, "all_cores_cores": 16})


def test_headline_is_the_last_line_and_compact():
    import io
    aux = {"aux_of": bench.METRIC, "aux": {"w%d" % k: {"gbps": 1.0, "note": "z" * 500} for k in range(60)}}
    buf = io.StringIO()
    bench.emit(aux, _headline(), out=buf)
    lines = buf.getvalue().splitlines()
    assert len(lines) == 2
    assert json.loads(lines[0])["aux_of"] == bench.METRIC
    last = lines[-1]
    assert len(last.encode()) < 4096
    d = json.loads(last)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks", "parity"):
        assert key in d, key
    assert d["config"]["workload"] and d["value"] == 7137.7
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in d["e2e"], key
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in d["cpu_baseline"], key
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0


def test_headline_refuses_to_grow_past_the_limit():
    import io
    with pytest.raises(RuntimeError):
        bench.emit(None, _headline(note_len=5000), out=io.StringIO())


def test_headline_withholds_value_on_mismatch():
    d = _headline(parity="MISMATCH")
    assert d["value"] is None and d["vs_baseline"] is None and d["parity"] == "MISMATCH"
    assert _headline(parity="unchecked")["value"] == 7137.7


def test_parity_windows_cover_head_tail_and_stay_in_range():
    assert bench.parity_windows(1000, 1) == [(0, 1000)]
    n = 1 << 28
    w = bench.parity_windows(n, 7)
    assert w[0] == (0, 1 << 20) and w[-1] == (n - (1 << 20), n)
    assert all(0 <= lo < hi <= n and hi - lo == 1 << 20 for lo, hi in w)
    assert len(w) >= 3
    assert bench.parity_windows(n, 7) == w  # seeded
    assert len(bench.parity_windows(33554432, 3, full_max=0)) >= 3


def test_first_mismatch_bits_and_nan_class():
    import numpy as np
    a = np.array([1.0, -0.0, np.nan], dtype=np.float32)
    b = a.copy()
    assert bench.first_mismatch(a, b, "f32", False) is None
    b[1] = 0.0  # -0 against +0 is a mismatch
    assert bench.first_mismatch(a, b, "f32", True) == 1
    c = a.copy()
    c.view(np.uint32)[2] = 0x7FC00001  # another NaN: a match only as a class
    assert bench.first_mismatch(a, c, "f32", True) is None
    assert bench.first_mismatch(a, c, "f32", False) == 2
    h = np.array([0x7E00, 0x3C00], dtype=np.uint16)
    g = np.array([0x7E01, 0x3C00], dtype=np.uint16)
    assert bench.first_mismatch(g, h, "f16", True) is None
    assert bench.first_mismatch(np.array([1, 2], np.int32), np.array([1, 3], np.int32), "i32", True) == 1


def test_nvml_summary_names_reasons():
    out = bench.summarize_nvml_samples([(2070.0, 0), (2040.0, 0x4), (2070.0, 0x0)], 2070.0)
    assert out["sm_mhz"] == 2070.0 and out["sm_mhz_min"] == 2040.0
    assert out["reasons"] == ["sw_power_cap"] and out["window"] == "timed region"
    hot = bench.summarize_nvml_samples([(1500.0, 0x40 | 0x8)], 2070.0)
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.summarize_nvml_samples([], 2070.0) is None


class _FakeNvml:
    """Stands in for libnvidia-ml: writes through the byref arguments."""

    def __init__(self):
        self.mhz = iter([2070, 2055, 2070])
        self.bits = iter([0, 0x4, 0])
        self.bus = None

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, h):
        self.bus = bus
        return 0

    def nvmlDeviceGetHandleByIndex_v2(self, i, h):
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        out._obj.value = next(self.mhz)
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = next(self.bits)
        return 0


def test_nvml_clocks_through_a_fake_library():
    fake = _FakeNvml()
    clk = bench.NvmlClocks("00000000:01:00.0", 0, lib=fake)
    assert clk.ok and fake.bus == b"00000000:01:00.0"
    for _ in range(3):
        clk.sample()
    s = clk.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_sectors_lookup_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    from memory_bound_elementwise_gb300 import _build
    prof = tmp_path / "profiles"
    prof.mkdir()
    ent = {"sectors_per_request": {"gather2_f32": 8.0, "copy_f32": 4.0, "metric": "m",
                                   "source_digest": _build.source_digest()}}
    (prof / "traffic.json").write_text(json.dumps(ent))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    got = bench.profiled_sectors()
    assert got["gather"] == 8.0 and got["copy"] == 4.0
    ent["sectors_per_request"]["source_digest"] = "0" * 64
    (prof / "traffic.json").write_text(json.dumps(ent))
    got = bench.profiled_sectors()
    assert got["gather"] is None and got["copy"] is None


class _FakeParity:
    """Stands in for the oracle comparison: reports a planted result."""

    def __init__(self, result):
        self.enabled = True
        self.result = result
        self.reruns = 0

    def check(self, name, out, want, n, **kw):
        return dict(self.result)


def _aux_with(parity):
    aux = bench.Aux.__new__(bench.Aux)  # only the bookkeeping of the entries is exercised
    aux.parity = parity
    aux.out = {}
    return aux


def test_parity_gate_drops_the_speed_of_a_mismatching_workload():
    aux = _aux_with(_FakeParity({"parity": "MISMATCH", "first_bad_index": 12345}))
    ran = []
    aux._finish("w", {"gbps": 7000.0, "frac": 1.03, "kernel_ms": 0.45}, (object(), None, 10, lambda: ran.append(1)))
    ent = aux.out["w"]
    assert ent["parity"] == "MISMATCH" and ent["first_bad_index"] == 12345
    assert "gbps" not in ent and "frac" not in ent and "kernel_ms" not in ent
    assert ran == [1]  # the in-place reset and relaunch ran before the comparison


def test_parity_gate_keeps_the_speed_of_a_matching_workload():
    aux = _aux_with(_FakeParity({"parity": True, "parity_elements": 10}))
    aux._finish("w", {"gbps": 7000.0}, (object(), None, 10))
    assert aux.out["w"]["gbps"] == 7000.0 and aux.out["w"]["parity"] is True
    aux._finish("lib", {"gbps": 6800.0}, None)
    assert aux.out["lib"]["parity"] == "not applicable" and aux.out["lib"]["gbps"] == 6800.0


def test_l2_resident_entries_carry_no_hbm_fraction():
    aux = _aux_with(None)
    aux.peak, aux.l2_bytes = 6796.2, 135528448

    class _M:
        @staticmethod
        def gbps(nbytes, s):
            return nbytes / s / 1e9
    aux.metrics = _M
    small = aux._speed(100663296, 8.1e-6)  # 2^23-element SAXPY: 100 MB per launch
    assert small["l2_resident"] is True and "frac" not in small and small["gbps"] > 10000
    big = aux._speed(402653184, 57e-6)
    assert "l2_resident" not in big and 1.0 < big["frac"] < 1.2


def test_gathers_are_compared_with_the_copy_of_their_own_dtype():
    out = {"copy_f32_2p26": {"gbps": 6500.0}, "copy_bf16_2p26": {"gbps": 6000.0},
           "gather12_f32_2p26": {"gbps": 6337.0},
           "gather2_bf16_2p26": {"gbps": 5980.0},
           "gather2_f32_2p26_index_order": {"gbps": 4680.0},
           "gather3_bf16_2p26": {"parity": "MISMATCH"},  # no speed: no fraction
           "add_f32_2p28": {"gbps": 7160.0}}
    bench.add_copy_fractions(out)
    assert out["gather12_f32_2p26"]["frac_of_copy_same_n"] == 6337.0 / 6500.0
    assert out["gather2_bf16_2p26"]["frac_of_copy_same_n"] == 5980.0 / 6000.0
    assert out["gather2_f32_2p26_index_order"]["frac_of_copy_same_n"] == 4680.0 / 6500.0
    assert "frac_of_copy_same_n" not in out["gather3_bf16_2p26"]
    assert "frac_of_copy_same_n" not in out["add_f32_2p28"]
    assert "frac_of_copy_same_n" not in out["copy_f32_2p26"]
