"""The C ABI on the host: symbols, argument validation and planning.

None of these calls reaches the GPU: every case is rejected (or planned) by
host code before any CUDA runtime call, so they run on a machine without one.
"""
import ctypes
import os
import re

import pytest

import memory_bound_elementwise_gb300 as ew
from tests.golden_util import load_golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(not os.path.exists(ew.LIB_PATH), reason="libew.so not built")

OK, INVALID, NULLP, DTYPE, OVERLAP = 0, 1, 2, 3, 4


def header_functions():
    with open(os.path.join(ROOT, "include", "ew.h"), encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"EW_API\s+[\w\s\*]+?\b(ew_\w+)\s*\(", text)))


def test_header_declares_the_expected_api():
    assert header_functions() == sorted(ew.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = ew.lib()
    for name in header_functions():
        assert hasattr(L, name), name
    assert L.ew_version() >= 100


def test_status_strings():
    for code, name in ew.STATUS_NAMES.items():
        assert ew.status_string(code).startswith(name)
    assert "unknown" in ew.status_string(99)


P = 0x10000000  # a fake, 256-byte aligned address: never dereferenced here


@pytest.mark.parametrize("dt", [0, 1, 2])
def test_zero_length_is_a_no_op(dt):
    L = ew.lib()
    assert L.ew_add(dt, None, None, None, 0, None) == OK
    assert L.ew_saxpy(dt, 2.5, None, None, 0, None) == OK
    assert L.ew_relu(dt, None, None, 0, None) == OK
    assert L.ew_add_relu(dt, None, None, None, 0, None) == OK
    assert L.ew_saxpy_relu(dt, 2.5, None, None, 0, None) == OK
    assert L.ew_select_even_odd(3, None, None, 0, None) == OK
    assert L.ew_copy(dt, None, None, 0, None) == OK
    assert L.ew_gather_stride(dt, None, None, 0, 2, None) == OK
    assert ew.last_launch()["launches"] == 0


def test_argument_errors_are_caught_on_the_host():
    L = ew.lib()
    assert L.ew_add(7, P, P + 4096, P + 8192, 10, None) == DTYPE
    assert L.ew_add(-1, P, P + 4096, P + 8192, 10, None) == DTYPE
    assert L.ew_add(0, P, P + 4096, P + 8192, -1, None) == INVALID
    assert L.ew_add(0, None, P + 4096, P + 8192, 10, None) == NULLP
    assert L.ew_add(0, P, None, P + 8192, 10, None) == NULLP
    assert L.ew_add(0, P, P + 4096, None, 10, None) == NULLP
    assert L.ew_saxpy(0, 2.5, None, P, 10, None) == NULLP
    assert L.ew_relu(1, P, None, 10, None) == NULLP
    assert L.ew_add_relu(0, P, P + 4096, None, 10, None) == NULLP
    assert L.ew_add_relu(4, P, P + 4096, P + 8192, 10, None) == DTYPE
    assert L.ew_add_relu(0, P, P + 4096, P + 4, 10, None) == OVERLAP
    assert L.ew_saxpy_relu(0, 2.5, P, None, 10, None) == NULLP
    assert L.ew_saxpy_relu(3, 2.5, P, P + 4096, 10, None) == DTYPE
    assert L.ew_saxpy_relu(0, 2.5, P, P + 4, 10, None) == OVERLAP
    assert L.ew_saxpy_relu(1, 2.5, P + 1, P + 4096, 10, None) == INVALID
    # int32 is taken by the select, copy and gather only
    assert L.ew_add(3, P, P + 4096, P + 8192, 10, None) == DTYPE
    assert L.ew_saxpy(3, 1.0, P, P + 4096, 10, None) == DTYPE
    assert L.ew_relu(3, P, P + 4096, 10, None) == DTYPE
    assert L.ew_add_relu(3, P, P + 4096, P + 8192, 10, None) == DTYPE
    assert L.ew_select_even_odd(0, P, P + 4096, 10, None) == DTYPE
    assert L.ew_select_even_odd(3, None, P + 4096, 10, None) == NULLP
    assert L.ew_select_even_odd(3, P, P + 4, 10, None) == OVERLAP
    assert L.ew_select_even_odd(3, P + 2, P + 4096, 10, None) == INVALID
    # misaligned to the element size
    assert L.ew_add(0, P + 2, P + 4096, P + 8192, 10, None) == INVALID
    assert L.ew_relu(2, P + 1, P + 4096, 10, None) == INVALID
    assert L.ew_copy(0, P, P + 4097, 10, None) == INVALID
    # gather stride must be positive
    assert L.ew_gather_stride(0, P, P + 4096, 10, 0, None) == INVALID
    assert L.ew_gather_stride(0, P, P + 4096, 10, -2, None) == INVALID
    assert L.ew_set_path(9) == INVALID
    assert L.ew_set_path(-1) == INVALID
    assert L.ew_set_pointer_check(2) == INVALID
    assert L.ew_set_schedule(5) == INVALID
    assert L.ew_set_schedule(-1) == INVALID
    assert L.ew_selftest_bounded_wait(0, None) == INVALID
    assert L.ew_selftest_bounded_wait(10 ** 11, None) == INVALID
    assert ew.last_launch()["launches"] == 0


def test_partial_overlap_is_rejected_identity_is_not_checked_as_overlap():
    L = ew.lib()
    n = 100
    # c overlaps a by one element
    assert L.ew_add(0, P, P + 4096, P + 4 * (n - 1), n, None) == OVERLAP
    assert L.ew_add(0, P + 4096, P, P + 4 * (n - 1), n, None) == OVERLAP
    assert L.ew_saxpy(0, 1.0, P, P + 4, n, None) == OVERLAP
    assert L.ew_relu(1, P, P + 2, n, None) == OVERLAP
    assert L.ew_copy(2, P + 2 * (n - 1), P, n, None) == OVERLAP
    # the gather accepts no overlap, not even identity
    assert L.ew_gather_stride(0, P, P, n, 2, None) == OVERLAP
    assert L.ew_gather_stride(0, P, P + 4 * (n - 1), n, 2, None) == OVERLAP
    # copy onto itself is a no-op that launches nothing
    assert L.ew_copy(0, P, P, n, None) == OK
    assert ew.last_launch()["launches"] == 0


def plan(dt, ptrs, n, path="auto"):
    ew.set_path(path)
    try:
        return ew.plan_query(dt, ptrs, n)
    finally:
        ew.set_path("auto")


def test_plan_aligned_f32_uses_256_bit_body():
    n = (1 << 20) + 3  # the odd-tail fp32 add size
    p = plan(0, [P, P + (1 << 24), P + (2 << 24)], n)
    assert p == {"path": 3, "vec_bytes": 32, "head": 0, "nvec": (1 << 20) // 8, "tail": 3}


def test_plan_offset_by_one_element_bf16():
    # all three pointers one bf16 element past a 256-byte boundary
    n = 1 << 28
    p = plan(2, [P + 2, P + 2 + (1 << 30), P + 2 + (2 << 30)], n)
    assert p["vec_bytes"] == 32 and p["head"] == 15
    assert p["head"] + p["nvec"] * 16 + p["tail"] == n
    assert p["tail"] == (n - 15) % 16


def test_plan_different_offsets_fall_back_to_shared_width():
    n = 1000
    # offsets 4, 0, 12 bytes: they agree modulo 4 only -> one element at a time
    assert plan(0, [P + 4, P, P + 12], n)["vec_bytes"] == 4
    # offsets 16, 0, 48: agree modulo 16 -> 128-bit body, head 0
    p = plan(0, [P + 16, P, P + 48], n)
    assert p["vec_bytes"] == 16 and p["head"] == 0
    # bf16 offsets 2 and 6 bytes: agree modulo 4 -> packed pairs after a 1-element head
    p = plan(2, [P + 2, P + 6], n)
    assert p["vec_bytes"] == 4 and p["head"] == 1 and p["nvec"] == (n - 1) // 2


def test_plan_bulk_copy_tiles():
    # 8 KiB tiles after a head that reaches 16-byte alignment
    n = (1 << 20) + 3
    p = plan(0, [P, P + (1 << 24), P + (2 << 24)], n, "tma")
    assert p == {"path": 4, "vec_bytes": 16, "head": 0, "nvec": n // 2048, "tail": n % 2048}
    p = plan(2, [P + 2, P + 2 + 4096, P + 2 + 8192], 100_000, "tma")
    assert p["path"] == 4 and p["head"] == 7
    assert p["head"] + p["nvec"] * 4096 + p["tail"] == 100_000
    # pointers that disagree modulo 16: the realigning kernel's tiles follow the
    # output (last pointer, 8 bytes past a 16-byte boundary): 2 elements reach
    # alignment, 4 more keep a 16-byte margin before the first staged span
    p = plan(0, [P + 4, P, P + 8], 100_000, "tma")
    assert p == {"path": 4, "vec_bytes": 16, "head": 6, "nvec": (100_000 - 6 - 4) // 2048,
                 "tail": 100_000 - 6 - (100_000 - 10) // 2048 * 2048}
    # too short for a tile with both margins: everything one by one
    p = plan(0, [P + 4, P, P + 8], 2048 + 9, "tma")
    assert p == {"path": 4, "vec_bytes": 16, "head": 6, "nvec": 0, "tail": 2048 + 3}


def test_plan_auto_realigns_16bit_parity_mismatch():
    # bf16 pointers of different parity take the realigning bulk-copy kernel
    # under AUTO from 2^22 elements; below that, 2-byte accesses
    n = 1 << 22
    p = plan(2, [P + 2, P, P + 6], n)
    assert p["path"] == 4 and p["vec_bytes"] == 16
    assert (P + 6 + p["head"] * 2) % 16 == 0 and p["head"] * 2 >= 16
    assert p["head"] + p["nvec"] * 4096 + p["tail"] == n and p["tail"] * 2 >= 16
    p = plan(2, [P + 2, P, P + 6], n - 1)
    assert p["path"] == 1 and p["vec_bytes"] == 2
    # same parity (4-byte accesses) and fp32 keep the vector kernels
    assert plan(2, [P + 2, P + 6, P + 10], n)["path"] != 4
    assert plan(0, [P + 4, P, P + 8], n)["path"] != 4
    # an explicit vector path never realigns
    assert plan(2, [P + 2, P, P + 6], n, "v256")["path"] == 1


def test_programmatic_launch_switch():
    L = ew.lib()
    assert L.ew_set_programmatic_launch(2) == INVALID
    assert L.ew_set_programmatic_launch(-1) == INVALID
    assert ew.get_programmatic_launch() is True  # on by default
    ew.set_programmatic_launch(False)
    assert ew.get_programmatic_launch() is False
    ew.set_programmatic_launch(True)
    assert ew.get_programmatic_launch() is True


def test_schedule_roundtrip():
    for name in ("oneshot", "persistent", "laps", "tiled", "auto"):
        ew.set_schedule(name)
        assert ew.get_schedule() == name


def test_plan_forced_widths():
    n = 1000
    ptrs = [P, P + 4096, P + 8192]
    assert plan(0, ptrs, n, "scalar") == {"path": 1, "vec_bytes": 4, "head": 0, "nvec": n, "tail": 0}
    assert plan(0, ptrs, n, "v128")["vec_bytes"] == 16
    assert plan(0, ptrs, n, "v256")["vec_bytes"] == 32


def test_plan_float4_worked_example():
    # the page's float4 loop: N = 10 gives 2 whole vectors and elements 8, 9 as tail
    case = load_golden("launch_geometry.json")["vector_tail"][0]
    p = plan(0, [P, P + 4096, P + 8192], case["n"], "v128")
    assert p["vec_bytes"] // 4 == case["elements_per_vector"]
    assert p["nvec"] == case["whole_vectors"]
    assert p["head"] == 0 and p["tail"] == len(case["tail_indices"])


@pytest.mark.parametrize("e,dt", [(4, 0), (2, 1), (2, 2)])
def test_plan_covers_every_size_and_offset(e, dt):
    for n in list(range(0, 70)) + [1000, 4099]:
        for off in range(0, 32, e):
            p = plan(dt, [P + off, P + 8192 + off], n)
            per = p["vec_bytes"] // e
            assert p["head"] + p["nvec"] * per + p["tail"] == n
            assert 0 <= p["tail"] < per or p["nvec"] == 0
            if p["nvec"] > 0:
                assert (P + off + p["head"] * e) % p["vec_bytes"] == 0


def test_plan_query_argument_errors():
    L = ew.lib()
    out = ew.Plan()
    arr = (ctypes.c_void_p * 1)(ctypes.c_void_p(P))
    assert L.ew_plan_query(0, arr, 0, 10, ctypes.byref(out)) == INVALID
    assert L.ew_plan_query(0, arr, 5, 10, ctypes.byref(out)) == INVALID
    assert L.ew_plan_query(0, None, 1, 10, ctypes.byref(out)) == NULLP
    assert L.ew_plan_query(0, arr, 1, 10, None) == NULLP
    assert L.ew_plan_query(5, arr, 1, 10, ctypes.byref(out)) == DTYPE


def test_binding_rejects_cpu_tensors():
    import torch
    a = torch.zeros(8)
    with pytest.raises(ValueError):
        ew.ew_add(a, a, torch.zeros(8))
