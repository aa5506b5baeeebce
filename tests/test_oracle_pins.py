"""Pins for the CPU oracle against facts fixed outside it.

Each test compares the oracle with something independent of its own code:
library conversions and arithmetic (numpy, torch), exact rational arithmetic,
closed forms on exactly representable values, invariants of the operations,
and brute force on tiny inputs.  A plausible slip in the oracle (a dropped
rounding step, a wrong exponent bias, a flipped comparison, a transposed
index) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_elementwise_gb300 import inputs
from tests import exact

ALL16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _f16_nan(bits):
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)


def _bf16_nan(bits):
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def _f32_nan(x):
    u = x.view(np.uint32)
    return (u & 0x7FFFFFFF) > 0x7F800000


# ---------------------------------------------------------------- formats


def test_f16_decode_all_patterns_match_numpy():
    got = oracle.decode_all("f16")
    ref = ALL16.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_all_patterns_match_bit_widening():
    got = oracle.decode_all("bf16")
    ref = (ALL16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_encode_roundtrips_every_pattern(dtype):
    dec = oracle.decode_all(dtype)
    enc = oracle.f64_to_f16 if dtype == "f16" else oracle.f64_to_bf16
    isnan = _f16_nan(ALL16) if dtype == "f16" else _bf16_nan(ALL16)
    for h in range(1 << 16):
        e = enc(dec[h])
        if isnan[h]:
            assert (_f16_nan if dtype == "f16" else _bf16_nan)(np.uint16(e))
        else:
            assert e == h, (dtype, hex(h), hex(e))


def test_f16_encode_matches_numpy_on_midpoints_and_neighbours():
    h = np.arange(0, 0x7BFF, dtype=np.uint16)  # every finite positive pattern but the max
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2  # exact in binary64
    probes = np.concatenate([mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf),
                             -mid, [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25,
                                    2.0 ** -25 * 1.0000001, 2.0 ** -26, 0.0, -0.0]])
    ref = probes.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_f16(p) for p in probes], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_matches_torch_on_random_binary32():
    x = inputs.random_bits(200_000, "f32", seed=11)
    x = x[~_f32_nan(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_encode_uses_bits_beyond_binary32():
    # mid-point between two bfloat16 neighbours, nudged by far less than a
    # binary32 ulp: only a correct sticky-bit decision rounds these right.
    for h in (0x3F80, 0x3F81, 0x0080, 0x4B7F, 0x0001, 0x7F7E):
        lo = float(np.uint32(h << 16).view(np.float32))
        hi = float(np.uint32((h + 1) << 16).view(np.float32))
        mid = (lo + hi) / 2
        tiny = (hi - lo) * 2.0 ** -40
        assert oracle.f64_to_bf16(mid + tiny) == h + 1
        assert oracle.f64_to_bf16(mid - tiny) == h
        assert oracle.f64_to_bf16(mid) == (h if h % 2 == 0 else h + 1)


def test_encode_overflow_and_underflow_thresholds():
    # binary16: max finite 65504, overflow threshold 65520 (tie to even -> inf)
    assert oracle.f64_to_f16(65504.0) == 0x7BFF
    assert oracle.f64_to_f16(np.nextafter(65520.0, 0)) == 0x7BFF
    assert oracle.f64_to_f16(65520.0) == 0x7C00
    assert oracle.f64_to_f16(-65520.0) == 0xFC00
    assert oracle.f64_to_f16(70000.0) == 0x7C00      # beyond the top binade: inf, not NaN
    assert oracle.f64_to_f16(-131000.0) == 0xFC00
    # smallest subnormal 2^-24; half of it ties to even (zero), a hair above rounds up
    assert oracle.f64_to_f16(2.0 ** -25) == 0x0000
    assert oracle.f64_to_f16(np.nextafter(2.0 ** -25, 1)) == 0x0001
    assert oracle.f64_to_f16(3 * 2.0 ** -25) == 0x0002
    assert oracle.f64_to_f16(-0.0) == 0x8000
    # bfloat16: max finite (2 - 2^-7) 2^127, threshold (2 - 2^-8) 2^127
    assert oracle.f64_to_bf16((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle.f64_to_bf16((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    assert oracle.f64_to_bf16(2.0 ** -134) == 0x0000
    assert oracle.f64_to_bf16(3 * 2.0 ** -134) == 0x0002
    assert oracle.f64_to_bf16(3.0 * 2.0 ** 127) == 0x7F80
    assert oracle.f64_to_bf16(-3.5 * 2.0 ** 128) == 0xFF80
    assert oracle.f64_to_bf16(math.inf) == 0x7F80
    assert oracle.f64_to_bf16(-math.inf) == 0xFF80


# ---------------------------------------------------------------- add


def test_add_f32_matches_numpy_binary32_addition():
    a = inputs.with_specials(inputs.uniform(300_001, 21), "f32", 21)
    b = inputs.with_specials(inputs.normal(300_001, 22) * np.float32(1e3), "f32", 22)
    a[:5000] = inputs.random_bits(5000, "f32", 23)
    with np.errstate(all="ignore"):
        ref = a + b
    got = oracle.add("f32", a, b)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_add_f32_closed_forms():
    k = np.arange(-4096, 4096, dtype=np.float32)
    got = oracle.add("f32", k, k[::-1].copy())
    assert np.array_equal(got, np.full_like(k, -1.0))
    # k * 2^-20 + 1 is exact for |k| < 2^20
    a = (np.arange(1, 1000, dtype=np.float32) * np.float32(2.0 ** -20)).astype(np.float32)
    got = oracle.add("f32", a, np.ones_like(a))
    assert np.array_equal(got, (1.0 + np.arange(1, 1000) * 2.0 ** -20).astype(np.float32))
    # 1 + 2^-24 is a tie and rounds to even (1); 1 + 3*2^-24 rounds up to 1 + 2^-22
    got = oracle.add("f32", np.float32([1.0, 1.0, 1.0]),
                     np.float32([2.0 ** -24, 3 * 2.0 ** -24, 2.0 ** -23]))
    assert got.tolist() == [1.0, 1.0 + 2.0 ** -22, 1.0 + 2.0 ** -23]
    # exact cancellation gives +0; (-0) + (-0) = -0
    got = oracle.add("f32", np.float32([1.5, -0.0]), np.float32([-1.5, -0.0]))
    assert got.view(np.uint32).tolist() == [0x00000000, 0x80000000]
    # overflow to infinity
    got = oracle.add("f32", np.float32([3.4e38]), np.float32([3.4e38]))
    assert np.isinf(got[0]) and got[0] > 0


def test_add_f32_commutative_and_independent():
    a = inputs.uniform(4099, 31)
    b = inputs.uniform(4099, 32)
    c = oracle.add("f32", a, b)
    assert np.array_equal(c.view(np.uint32), oracle.add("f32", b, a).view(np.uint32))
    # output j depends only on a[j], b[j]
    a2 = a.copy()
    a2[1234] = np.float32(7.0)
    c2 = oracle.add("f32", a2, b)
    diff = np.nonzero(c2.view(np.uint32) != c.view(np.uint32))[0]
    assert diff.tolist() == [1234]


@pytest.mark.parametrize("n", list(range(0, 40)) + [255, 256, 257, 300])
def test_add_f32_brute_force_tiny(n):
    a = inputs.uniform(n, 100 + n) * np.float32(3.0)
    b = inputs.normal(n, 200 + n)
    got = oracle.add("f32", a, b)
    for i in range(n):
        assert got[i] == exact.to_f32(exact.frac(a[i]) + exact.frac(b[i]))


def test_add_f16_matches_numpy_half_arithmetic_structured_sample():
    # every binary16 pattern as A against 512 seeded patterns as B
    bvals = inputs.random_bits(512, "f16", 41)
    bvals[:20] = inputs.SPECIAL_BITS["f16"]
    for chunk in np.array_split(bvals, 8):
        A = np.repeat(ALL16[None, :], chunk.size, axis=0).ravel()
        B = np.repeat(chunk, ALL16.size)
        got = oracle.add("f16", A, B)
        with np.errstate(all="ignore"):
            ref = (A.view(np.float16) + B.view(np.float16)).view(np.uint16)
        nan = _f16_nan(ref)
        assert np.array_equal(_f16_nan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def test_add_bf16_matches_torch_bfloat16_arithmetic_structured_sample():
    bvals = inputs.random_bits(512, "bf16", 42)
    bvals[:20] = inputs.SPECIAL_BITS["bf16"]
    for chunk in np.array_split(bvals, 8):
        A = np.repeat(ALL16[None, :], chunk.size, axis=0).ravel()
        B = np.repeat(chunk, ALL16.size)
        got = oracle.add("bf16", A, B)
        ta = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16)
        tb = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16)
        ref = (ta + tb).view(torch.int16).numpy().view(np.uint16)
        nan = _bf16_nan(ref)
        assert np.array_equal(_bf16_nan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_add_16bit_equals_exact_rounding_on_sample(dtype):
    # correctly rounded sum via exact rationals and the format definition
    a = inputs.as_dtype(inputs.normal(3000, 51) * np.float32(100), dtype)
    b = inputs.as_dtype(inputs.normal(3000, 52) * np.float32(0.01), dtype)
    got = oracle.add(dtype, a, b)
    bits, emin, emax = (11, -14, 15) if dtype == "f16" else (8, -126, 127)
    dec = oracle.f16_to_f64 if dtype == "f16" else oracle.bf16_to_f64
    for i in range(a.size):
        q = exact.frac(dec(a[i])) + exact.frac(dec(b[i]))
        want = exact.round_binary(q, bits, emin, emax)
        assert dec(got[i]) == float(want), (dtype, i)


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_add_16bit_exhaustive_all_pairs(dtype):
    for hb in range(1 << 16):
        B = np.full(1 << 16, hb, dtype=np.uint16)
        got = oracle.add(dtype, ALL16, B)
        if dtype == "f16":
            with np.errstate(all="ignore"):
                ref = (ALL16.view(np.float16) + B.view(np.float16)).view(np.uint16)
            nan = _f16_nan(ref)
        else:
            ta = torch.from_numpy(ALL16.view(np.int16)).view(torch.bfloat16)
            tb = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16)
            ref = (ta + tb).view(torch.int16).numpy().view(np.uint16)
            nan = _bf16_nan(ref)
        assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- saxpy


def test_saxpy_f32_equals_exact_fused_rounding():
    n = 20_000
    x = inputs.normal(n, 61)
    y = inputs.normal(n, 62)
    x[:100] *= np.float32(1e-30)   # small products: y dominates
    y[100:200] *= np.float32(1e-30)  # small y: product dominates
    # alpha is a binary32 argument: the exact reference must use the same value
    for alpha in (np.float32(2.5), np.float32(-1 / 3), np.float32(1e-3)):
        got = oracle.saxpy("f32", float(alpha), x, y)
        for i in range(n):
            assert got[i] == exact.exact_fma_f32(alpha, x[i], y[i]), (alpha, i)


def test_saxpy_f32_differs_from_unfused_somewhere():
    # a fused multiply-add rounds once; the unfused form rounds twice.  Over
    # many random operands the two must disagree at least once.
    x = inputs.normal(100_000, 63)
    y = inputs.normal(100_000, 64)
    got = oracle.saxpy("f32", 2.5, x, y)
    unfused = (np.float32(2.5) * x + y).astype(np.float32)
    assert np.any(got != unfused)


def test_saxpy_special_cases():
    x = inputs.normal(1000, 65)
    y = inputs.normal(1000, 66)
    assert np.array_equal(oracle.saxpy("f32", 0.0, x, y), y)           # alpha = 0
    assert np.array_equal(oracle.saxpy("f32", 2.5, np.zeros_like(x), y), y)  # x = 0
    z = oracle.saxpy("f32", 2.5, x, np.zeros_like(y))                   # y = 0
    assert np.array_equal(z, (np.float32(2.5) * x).astype(np.float32))
    # the pages' SAXPY size and alpha: in-place form leaves x untouched
    xs = x.copy()
    oracle.saxpy("f32", 2.5, x, y)
    assert np.array_equal(xs, x)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_saxpy_16bit_is_fused_binary32_then_one_rounding(dtype):
    x = inputs.as_dtype(inputs.normal(4000, 67), dtype)
    y = inputs.as_dtype(inputs.normal(4000, 68), dtype)
    dec = oracle.f16_to_f64 if dtype == "f16" else oracle.bf16_to_f64
    got = oracle.saxpy(dtype, 2.5, x, y)
    r32 = np.array([exact.exact_fma_f32(2.5, dec(x[i]), dec(y[i])) if
                    (2.5 * dec(x[i]) + dec(y[i])) != 0 else np.float32(0)
                    for i in range(x.size)], dtype=np.float32)
    assert np.array_equal(got, inputs.as_dtype(r32, dtype))


# ---------------------------------------------------------------- relu


def _relu_properties(dtype, x, y):
    if dtype == "f32":
        xb, yb = x.view(np.uint32), y.view(np.uint32)
        nan = _f32_nan(x)
        sign = np.uint32(0x80000000)
        pos = (~nan) & ((xb & sign) == 0) & (xb != 0)
    else:
        xb, yb = x, y
        nan = _f16_nan(x) if dtype == "f16" else _bf16_nan(x)
        sign = np.uint16(0x8000)
        pos = (~nan) & ((xb & sign) == 0) & (xb != 0)
    # NaN passes through bit for bit; x > 0 passes through; everything else is +0
    assert np.array_equal(yb[nan], xb[nan])
    assert np.array_equal(yb[pos], xb[pos])
    assert np.all(yb[~nan & ~pos] == 0)
    # sign bit clear on every non-NaN output; zero count == count of x <= 0
    assert np.all((yb[~nan] & sign) == 0)
    assert int(np.sum(yb[~nan] == 0)) == int(np.sum(~nan & ~pos))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_relu_16bit_every_pattern(dtype):
    y = oracle.relu(dtype, ALL16)
    _relu_properties(dtype, ALL16, y)
    assert np.array_equal(oracle.relu(dtype, y), y)  # idempotent


def test_relu_f32_random_patterns_and_zeros():
    x = inputs.random_bits(500_000, "f32", 71)
    x[:1000] = inputs.normal(1000, 72)
    inputs.inject_signed_zeros(x, period=97)
    y = oracle.relu("f32", x)
    _relu_properties("f32", x, y)
    assert np.array_equal(oracle.relu("f32", y).view(np.uint32), y.view(np.uint32))
    xi = x.copy()
    oracle.relu_inplace("f32", xi)
    assert np.array_equal(xi.view(np.uint32), y.view(np.uint32))
    # numeric values agree with max(x, 0) wherever x is not NaN
    nan = _f32_nan(x)
    assert np.array_equal(y[~nan], np.maximum(x[~nan], np.float32(0)))


def test_relu_signed_zero_reading():
    y = oracle.relu("f32", np.float32([-0.0, 0.0, -1e-45, 1e-45]))
    assert y.view(np.uint32).tolist() == [0, 0, 0, 1]


# ---------------------------------------------------------------- copy, gather


def test_copy_is_bitwise():
    for dtype, n in (("f32", 1001), ("f16", 77), ("bf16", 4096)):
        x = inputs.random_bits(n, dtype, 81)
        y = oracle.copy(x)
        assert y.tobytes() == x.tobytes()


@pytest.mark.parametrize("n", list(range(1, 34)) + [64, 100, 1001])
@pytest.mark.parametrize("s", [1, 2, 3, 5, 7, 1 << 40])
def test_gather_brute_force_tiny(n, s):
    x = inputs.random_bits(n, "f32", 90 + n)
    got = oracle.gather_stride(x, s)
    xb = x.view(np.uint32)
    want = [int(xb[(s * i) % n]) for i in range(n)]
    assert got.view(np.uint32).tolist() == want


def test_gather_stride2_structure():
    n = 1 << 12
    x = inputs.random_bits(n, "f32", 91)
    y = oracle.gather_stride(x, 2).view(np.uint32)
    xb = x.view(np.uint32)
    h = n // 2
    assert np.array_equal(y[:h], y[h:])          # even n: the map wraps after n/2
    assert np.array_equal(y[:h], xb[0::2])       # and reads the even-indexed inputs
    n = 4097                                      # odd n: (2i) mod n is a permutation
    x = inputs.random_bits(n, "f32", 92)
    y = oracle.gather_stride(x, 2).view(np.uint32)
    assert np.array_equal(np.sort(y), np.sort(x.view(np.uint32)))


def test_gather_index_no_overflow():
    big = (1 << 62) + 12345
    for i, s, n in ((big, 3, (1 << 61) - 1), ((1 << 63) - 1, (1 << 63) - 1, 1000003),
                    (5, 2, 7), (0, 9, 1)):
        assert oracle.gather_index(i, s, n) == (i * s) % n


# ---------------------------------------------------------------- select


def test_select_even_odd_closed_forms_and_wrap():
    x = np.array([0, 1, 2, 3, -1, -2, -3, 7, 2 ** 31 - 1, -2 ** 31, 2 ** 30, 2 ** 30 + 1],
                 dtype=np.int32)
    want = [0, 2, 4, 4, 0, -4, -2, 8, -2 ** 31, 0, -2 ** 31, 2 ** 30 + 2]
    assert oracle.select_even_odd(x).tolist() == want


def test_select_even_odd_brute_force():
    g = inputs.rng(1234)
    x = g.integers(-2 ** 31, 2 ** 31, size=100_000, dtype=np.int64).astype(np.int32)
    got = oracle.select_even_odd(x)
    for v, r in zip(x[:20000].tolist(), got[:20000].tolist()):
        w = (2 * v) if v % 2 == 0 else (v + 1)
        w = (w + 2 ** 31) % 2 ** 32 - 2 ** 31  # two's complement wrap
        assert r == w
    # parity: even inputs give even results that are twice the input (mod 2^32)
    even = (x % 2 == 0)
    assert np.array_equal(got[even].astype(np.int64) % 2, np.zeros(int(even.sum()), np.int64))
    assert np.array_equal(got[~even], (x[~even].astype(np.int64) + 1).astype(np.int32))
