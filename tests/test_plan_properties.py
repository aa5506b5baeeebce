"""Property tests of the host-side planner (hypothesis; no GPU involved)."""
import os

import pytest

import memory_bound_elementwise_gb300 as ew

try:  # the property test needs hypothesis; without it the test is skipped, not the module
    from hypothesis import given, settings, strategies as st
except ImportError:
    given = None

pytestmark = pytest.mark.skipif(not os.path.exists(ew.LIB_PATH), reason="libew.so not built")

BASE = 0x7f0000000000  # fake, 4 KiB aligned; never dereferenced
ESIZE = {0: 4, 1: 2, 2: 2}
CAP = {"scalar": None, "v128": 16, "v256": 32, "auto": 32, "tma": 32}


def _cap(path, e, n):
    """Widest access a path may use."""
    return CAP[path] or e


def _property(test):
    if given is None:
        @pytest.mark.skip(reason="hypothesis is not installed")
        def skipped():
            pass
        return skipped
    return settings(max_examples=400, deadline=None)(given(
        dt=st.sampled_from([0, 1, 2]),
        n=st.one_of(st.integers(0, 100), st.integers(0, 1 << 40)),
        offsets=st.lists(st.integers(0, 63), min_size=1, max_size=4),
        path=st.sampled_from(["auto", "scalar", "v128", "v256", "tma"]))(test))


@_property
def test_plan_partitions_and_aligns(dt, n, offsets, path):
    e = ESIZE[dt]
    ptrs = [BASE + (k << 34) + o * e for k, o in enumerate(offsets)]
    ew.set_path(path)
    try:
        p = ew.plan_query(dt, ptrs, n)
    finally:
        ew.set_path("auto")
    vb = p["vec_bytes"]
    same16 = len({q % 16 for q in ptrs}) == 1
    if p["path"] == 4:  # bulk copy: 8 KiB tiles after a 16-byte aligned head
        per = 8192 // e
        assert vb == 16
        assert path == "tma" or (path == "auto" and e == 2 and n >= 1 << 22
                                 and len({q % 4 for q in ptrs}) > 1)
    else:
        per = vb // e
        cap = _cap(path, e, n)
        assert e <= vb <= cap and (vb & (vb - 1)) == 0
    assert p["head"] + p["nvec"] * per + p["tail"] == n
    assert p["head"] >= 0 and p["tail"] >= 0 and p["nvec"] >= 0
    if p["nvec"] > 0:
        if p["path"] == 4 and not same16:
            # realigning bulk copy: the output (last pointer) is aligned, and
            # 16 bytes stay outside the tiles at both ends
            assert (ptrs[-1] + p["head"] * e) % 16 == 0
            assert p["head"] * e >= 16 and p["tail"] * e >= 16
            assert p["tail"] < per + 16 // e  # less than a tile beyond the end margin
        else:
            # every pointer reaches the vector boundary at the same element
            align = 16 if p["path"] == 4 else vb
            for q in ptrs:
                assert (q + p["head"] * e) % align == 0
            assert p["tail"] < per
    # the width is the widest the pointers share
    if p["path"] != 4 and vb < _cap(path, e, n):
        w = vb * 2
        assert len({q % w for q in ptrs}) > 1
