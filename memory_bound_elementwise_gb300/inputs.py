"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws numbers; it holds none of the operators' arithmetic.
Both the CUDA path and the CPU oracle receive the arrays it returns.

Random source: numpy's ``Generator(PCG64(seed))``.  Distributions follow the
pages' workloads, which draw ``torch.randn`` tensors ("HyperAI elementwise add
on RTX 5090", benchmark script) and 32M-element SAXPY vectors ("Puzzle 31"):

* ``uniform``  -- binary32 uniform on [lo, hi): ``lo + (hi-lo)*u`` with
  ``u = Generator.random(dtype=float32)`` (a multiple of 2^-24 in [0, 1)).
  For [-1, 1) the value ``2u - 1`` is exact in binary32.
* ``normal``   -- binary32 standard normal, ``Generator.standard_normal``.
* 16-bit inputs are binary32 draws rounded to the format, nearest-even, by
  library conversions (numpy ``astype(float16)``, torch ``to(bfloat16)``);
  they are stored and passed as ``uint16`` bit patterns.
"""
import numpy as np

SEED_BASE = 0xE1E00000

# config ids used to derive seeds; one per workload family
CONFIG_IDS = {
    "add_f32_small": 1,     # fp32 add, N = 2^20 + 3
    "saxpy_f32": 2,         # fp32 SAXPY, N = 32 * 2^20
    "add_16": 3,            # bf16 / fp16 add, N = 2^28
    "relu_f32": 4,          # fp32 ReLU, N = 2^28
    "copy_f32": 5,          # fp32 copy / stride-2 gather, N = 2^26
    "add_f32": 6,           # fp32 add, N = 2^28 (headline measurement)
}


def seed_for(config: str, stream: int = 0) -> int:
    return SEED_BASE + CONFIG_IDS[config] + (stream << 8)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(n: int, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    u = rng(seed).random(n, dtype=np.float32)
    if lo == 0.0 and hi == 1.0:
        return u
    return (np.float32(lo) + np.float32(hi - lo) * u).astype(np.float32)


def normal(n: int, seed: int) -> np.ndarray:
    return rng(seed).standard_normal(n, dtype=np.float32)


def to_f16_bits(x32: np.ndarray) -> np.ndarray:
    """Round binary32 values to binary16 (nearest-even); return bit patterns."""
    return np.ascontiguousarray(x32, dtype=np.float32).astype(np.float16).view(np.uint16)


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round binary32 values to bfloat16 (nearest-even); return bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def as_dtype(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Storage array of ``dtype`` ('f32', 'f16', 'bf16') holding x32 rounded."""
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "f16":
        return to_f16_bits(x32)
    if dtype == "bf16":
        return to_bf16_bits(x32)
    raise ValueError(dtype)


def inject_signed_zeros(x: np.ndarray, period: int = 4099) -> np.ndarray:
    """ReLU workload: x[0] = +0, x[1] = -0, and +-0 alternating every
    ``period``-th index (in place on a binary32 array)."""
    assert x.dtype == np.float32
    if x.size > 0:
        x[0] = np.float32(0.0)
    if x.size > 1:
        x[1] = np.float32(-0.0)
    idx = np.arange(period, x.size, period)
    x[idx[0::2]] = np.float32(0.0)
    x[idx[1::2]] = np.float32(-0.0)
    return x


# Bit patterns of special values, per storage type, for edge-case inputs.
SPECIAL_BITS = {
    "f32": np.array([
        0x00000000, 0x80000000,            # +0, -0
        0x00000001, 0x80000001,            # smallest subnormals
        0x007fffff, 0x807fffff,            # largest subnormals
        0x00800000, 0x80800000,            # smallest normals
        0x7f7fffff, 0xff7fffff,            # largest finite
        0x7f800000, 0xff800000,            # +-inf
        0x7fc00000, 0xffc00000,            # quiet NaNs
        0x7f800001, 0x7fa5a5a5,            # NaNs with payload
        0x3f800000, 0xbf800000,            # +-1
        0x33800000, 0x4b800000,            # 2^-24, 2^24
    ], dtype=np.uint32),
    "f16": np.array([
        0x0000, 0x8000, 0x0001, 0x8001, 0x03ff, 0x83ff, 0x0400, 0x8400,
        0x7bff, 0xfbff, 0x7c00, 0xfc00, 0x7e00, 0xfe00, 0x7c01, 0x7d55,
        0x3c00, 0xbc00, 0x1400, 0x6400,
    ], dtype=np.uint16),
    "bf16": np.array([
        0x0000, 0x8000, 0x0001, 0x8001, 0x007f, 0x807f, 0x0080, 0x8080,
        0x7f7f, 0xff7f, 0x7f80, 0xff80, 0x7fc0, 0xffc0, 0x7f81, 0x7fa5,
        0x3f80, 0xbf80, 0x3380, 0x4b80,
    ], dtype=np.uint16),
}


def with_specials(x: np.ndarray, dtype: str, seed: int, frac: float = 0.05) -> np.ndarray:
    """Overwrite a seeded random ``frac`` of positions with special values
    (signed zeros, subnormals, extremes, infinities, NaNs)."""
    x = np.array(x, copy=True)
    if x.size == 0:
        return x
    g = rng(seed ^ 0x5BEC)
    k = max(1, int(x.size * frac))
    pos = g.integers(0, x.size, size=k)
    bits = SPECIAL_BITS[dtype]
    vals = bits[g.integers(0, bits.size, size=k)]
    if dtype == "f32":
        x.view(np.uint32)[pos] = vals
    else:
        x[pos] = vals
    return x


def random_bits(n: int, dtype: str, seed: int) -> np.ndarray:
    """Uniformly random bit patterns (every encoding, NaNs included)."""
    g = rng(seed)
    if dtype == "f32":
        return g.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    return g.integers(0, 1 << 16, size=n, dtype=np.uint32).astype(np.uint16)
