"""Worked examples printed on the pages (fixtures under tests/golden/)."""
import pytest

import oracle
from memory_bound_elementwise_gb300 import metrics
from tests.golden_util import load_golden as load


def test_ceil_div_worked_example():
    for case in load("launch_geometry.json")["ceil_div"]:
        n, t = case["n"], case["threads_per_block"]
        blocks = oracle.ceil_div(n, t)
        assert blocks == case["blocks"]
        assert blocks * t == case["threads_total"]
        assert blocks * t - n == case["masked_threads"]
        assert (blocks - 1) * t < n <= blocks * t


def test_ceil_div_covers_all_sizes():
    for t in (1, 32, 256, 1024):
        for n in range(0, 3000, 7):
            b = oracle.ceil_div(n, t)
            assert b * t >= n and (b == 0 or (b - 1) * t < n)


def test_vector_tail_worked_example():
    for case in load("launch_geometry.json")["vector_tail"]:
        n, w = case["n"], case["elements_per_vector"]
        assert n // w == case["whole_vectors"]
        assert (n // w) * w == case["vector_elements"]
        assert list(range((n // w) * w, n)) == case["tail_indices"]


def test_bytes_per_element_add():
    g = load("traffic.json")["add_f32"]
    assert metrics.algorithmic_bytes("add", "f32", 1) == g["bytes_per_element"]
    assert metrics.arithmetic_intensity("add", "f32") == pytest.approx(g["intensity_flop_per_byte"], abs=5e-4)
    f = load("traffic.json")["benchmark_formula"]
    for dtype, e in (("f32", 4), ("f16", 2), ("bf16", 2)):
        assert metrics.algorithmic_bytes("add", dtype, 1000) == f["transfers_per_element"] * 1000 * e


def test_saxpy_traffic_32M():
    g = load("traffic.json")["saxpy_f32_32M"]
    b = metrics.algorithmic_bytes("saxpy", "f32", g["n"])
    assert b == g["total_mib"] * 2 ** 20
    assert g["n"] * 4 * 2 == g["read_mib"] * 2 ** 20 and g["n"] * 4 == g["write_mib"] * 2 ** 20
    # the page divides its 384 "MB" by 600 GB/s
    assert g["total_mib"] * 1e6 / (g["peak_gbps"] * 1e9) * 1e3 == pytest.approx(g["min_time_ms"], rel=1e-9)


def test_relu_intensity():
    g = load("traffic.json")["relu_f32"]
    assert metrics.algorithmic_bytes("relu", "f32", 1) == g["bytes_per_element_with_write"]
    assert metrics.arithmetic_intensity("relu", "f32") == pytest.approx(g["intensity_with_write"])
    assert 1 / g["bytes_per_element_no_write"] == pytest.approx(g["intensity_no_write"])


def test_bandwidth_formula_reproduces_rtx5090_table():
    for row in load("rtx5090_add_bandwidth.json")["rows"]:
        nbytes = metrics.algorithmic_bytes("add", row["dtype"], row["n"])
        got = metrics.gbps(nbytes, row["ms"] / 1e3)
        # printed ms has 4 decimals and printed GB/s has 1
        tol = row["gbps"] * (0.00005 / row["ms"]) * 1.01 + 0.05
        assert abs(got - row["gbps"]) <= tol, (row, got)
