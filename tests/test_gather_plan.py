"""Host-side gather planning (ew_gather_plan_query, no GPU involved): which
kernel schedule AUTO and the forced schedules pick for every stride from 1 to
70, both element sizes, input offsets within 16 bytes and ragged sizes, and
the launch geometry each plan reports, against an independent statement of
the rules (tests/gather_geometry.py)."""
import os

import pytest

import memory_bound_elementwise_gb300 as ew
from tests.gather_geometry import fixed_geometry, fixed_positions, general_positions, pow2_positions

pytestmark = pytest.mark.skipif(not os.path.exists(ew.LIB_PATH), reason="libew.so not built")

BASE = 0x7f0000000000  # fake, 4 KiB aligned; the query reads neither buffer
OUT = BASE + (1 << 40)
SCHED = {"oneshot": 1, "persistent": 2, "laps": 3, "tiled": 4}
LAP_BLOCK = 256 * 8      # outputs per lap-order block
ONESHOT_BLOCK = 256 * 4  # outputs per index-order block


def _pow2(s):
    return s & (s - 1) == 0


def _expected(e, n, stride, in_off, sched):
    """(schedule, kernel, lap positions per block or None) the rules give."""
    s = stride % n
    small = 2 <= s <= 64
    if n > 1 << 32 or sched == "persistent":
        return 2, "stride", None
    tiled = small and (sched == "tiled" or (sched == "auto" and s >= (2 if e == 2 else 5)))
    if tiled:
        aligned = (in_off * e) % 16 == 0
        if aligned and _pow2(s):
            return 4, "pow2", pow2_positions(s, e)
        if not _pow2(s) or (e == 2 and s <= 8):
            return 4, "fixed", fixed_positions(s, e)
        return 4, "general", general_positions(s, e)
    if sched != "oneshot" and small and n // s >= LAP_BLOCK:
        return 3, "laps", None
    return 1, "oneshot", None


def _check(dt, e, n, stride, in_off, sched, out=OUT):
    rec = ew.gather_plan_query(dt, BASE + in_off * e, out, n, stride)
    schedule, kernel, p = _expected(e, n, stride, in_off, sched)
    where = (dt, n, stride, in_off, sched, rec)
    assert rec["launches"] == 1 and rec["schedule"] == schedule, where
    s = stride % n
    lap_len = -(-n // s) if s else n
    if kernel == "laps":
        assert rec["block"] == 256 and rec["vec_bytes"] == e, where
        assert rec["grid"] == s * -(-lap_len // LAP_BLOCK), where
    elif kernel == "oneshot":
        assert rec["block"] == 256 and rec["vec_bytes"] == e, where
        assert rec["grid"] == -(-n // ONESHOT_BLOCK), where
    elif kernel == "stride":
        assert rec["grid"] == 0 and rec["vec_bytes"] == e, where  # depends on the device
    else:  # the tiled kernels: 16-byte staging, one block per P lap positions
        assert rec["path"] == 2 and rec["vec_bytes"] == 16, where
        assert rec["grid"] == -(-lap_len // p), where
        if kernel == "fixed":
            t, _ = fixed_geometry(s, e)
            assert rec["block"] == t, where
            pad = rec["smem"] // (s * e) - p  # rows of P positions plus a pad below 32 elements
            assert rec["smem"] == s * (p + pad) * e and 0 <= pad < 32 and (e == 4 or pad % 2 == 0), where
        else:
            assert rec["block"] == 256, where
            assert rec["smem"] >= s * p * e, where


@pytest.mark.parametrize("sched", ["auto", "tiled", "laps", "oneshot", "persistent"])
@pytest.mark.parametrize("dt,e", [(0, 4), (2, 2)])
def test_gather_plans_every_stride(dt, e, sched):
    ew.set_schedule(sched)
    try:
        for stride in range(1, 71):
            for n in (stride + 1, 4099, 300_007, 1 << 26, (1 << 26) + 13):
                for in_off in range(16 // e):
                    _check(dt, e, n, stride, in_off, sched)
    finally:
        ew.set_schedule("auto")


def test_gather_plans_strides_congruent_mod_n_and_huge_n():
    """A stride is taken mod n; above 2^32 elements the grid-stride kernel runs
    whatever the stride (its grid is the device's to decide: 0 here)."""
    n = 1 << 20
    for s in (3, 12, 64):
        assert ew.gather_plan_query(0, BASE, OUT, n, s) == ew.gather_plan_query(0, BASE, OUT, n, s + 5 * n)
    rec = ew.gather_plan_query(0, BASE, OUT, (1 << 32) + 1, 12)
    assert rec["schedule"] == 2 and rec["grid"] == 0 and rec["nvec"] == (1 << 32) + 1


def test_gather_plan_query_arguments():
    """The same checks as ew_gather_stride: n == 0 plans nothing, and bad
    arguments give the call's status."""
    assert ew.gather_plan_query(0, BASE, OUT, 0, 3)["launches"] == 0
    L = ew.lib()
    rec = ew.LaunchRecord()
    assert L.ew_gather_plan_query(0, BASE, OUT, 100, 0, rec) == 1            # stride <= 0
    assert L.ew_gather_plan_query(0, BASE, OUT, -1, 3, rec) == 1             # n < 0
    assert L.ew_gather_plan_query(0, BASE + 2, OUT, 100, 3, rec) == 1        # not element-aligned
    assert L.ew_gather_plan_query(0, 0, OUT, 100, 3, rec) == 2               # null input
    assert L.ew_gather_plan_query(0, BASE, OUT, 100, 3, None) == 2           # null record
    assert L.ew_gather_plan_query(9, BASE, OUT, 100, 3, rec) == 3            # dtype
    assert L.ew_gather_plan_query(0, BASE, BASE + 40, 100, 3, rec) == 4      # overlap


try:  # the property test needs hypothesis; without it that test alone is skipped
    from hypothesis import given, settings, strategies as st
except ImportError:
    given = None


def _property(test):
    if given is None:
        @pytest.mark.skip(reason="hypothesis is not installed")
        def skipped():
            pass
        return skipped
    return settings(max_examples=600, deadline=None)(given(
        dt=st.sampled_from([0, 1, 2, 3]),
        n=st.one_of(st.integers(1, 5000), st.integers(1, 1 << 33), st.integers(1, 1 << 40)),
        stride=st.one_of(st.integers(1, 80), st.integers(1, 1 << 41)),
        in_off=st.integers(0, 7),
        sched=st.sampled_from(["auto", "tiled", "laps", "oneshot", "persistent"]))(test))


@_property
def test_gather_plan_properties(dt, n, stride, in_off, sched):
    """Random sizes up to 2^40, strides up to 2^41 (taken mod n), input offsets
    and schedules: the plan follows the same rules."""
    e = 4 if dt in (0, 3) else 2
    in_off %= 16 // e
    ew.set_schedule(sched)
    try:
        _check(dt, e, n, stride, in_off, sched, out=BASE + (1 << 43))  # clear of n * e <= 2^42 bytes
    finally:
        ew.set_schedule("auto")
