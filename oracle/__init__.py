"""Python access to the C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain CPU definition of every
operator that the CUDA library implements.  Only the test suite, the package
smoke check and the benchmark's CPU-baseline leg may import this module.  It
never imports the product package, and the product package never imports it.

All functions take and return numpy arrays.  16-bit formats are passed as
``uint16`` bit patterns (IEEE binary16 for ``"f16"``, bfloat16 for ``"bf16"``);
binary32 as ``float32``.
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None

_F32P = ctypes.POINTER(ctypes.c_float)
_U16P = ctypes.POINTER(ctypes.c_uint16)
_I64 = ctypes.c_int64


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        for name in ("orc_add_f32",):
            getattr(L, name).argtypes = [_F32P, _F32P, _F32P, _I64]
        for name in ("orc_add_f16", "orc_add_bf16"):
            getattr(L, name).argtypes = [_U16P, _U16P, _U16P, _I64]
        L.orc_saxpy_f32.argtypes = [ctypes.c_float, _F32P, _F32P, _I64]
        for name in ("orc_saxpy_f16", "orc_saxpy_bf16"):
            getattr(L, name).argtypes = [ctypes.c_float, _U16P, _U16P, _I64]
        L.orc_relu_f32.argtypes = [_F32P, _F32P, _I64]
        for name in ("orc_relu_f16", "orc_relu_bf16"):
            getattr(L, name).argtypes = [_U16P, _U16P, _I64]
        L.orc_select_even_odd_i32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64]
        L.orc_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64, _I64]
        L.orc_gather_stride.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I64, _I64, _I64]
        L.orc_gather_index.argtypes = [_I64, _I64, _I64]
        L.orc_gather_index.restype = _I64
        L.orc_ceil_div.argtypes = [_I64, _I64]
        L.orc_ceil_div.restype = _I64
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_f64_to_f16.argtypes = [ctypes.c_double]
        L.orc_f64_to_f16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        _lib = L
    return _lib


DTYPES = ("f32", "f16", "bf16")
_NP_STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2}


def _arr(x, dtype):
    want = _NP_STORAGE[dtype]
    x = np.ascontiguousarray(x)
    if x.dtype != want:
        raise TypeError("oracle %s expects %s storage, got %s" % (dtype, want, x.dtype))
    return x


def _ptr(x, dtype):
    return x.ctypes.data_as(_F32P if dtype == "f32" else _U16P)


def add(dtype, a, b):
    """C = A + B, elementwise, one rounding to the storage type."""
    a, b = _arr(a, dtype), _arr(b, dtype)
    if a.shape != b.shape:
        raise ValueError("shape mismatch")
    c = np.empty_like(a)
    getattr(lib(), "orc_add_" + dtype)(_ptr(a, dtype), _ptr(b, dtype), _ptr(c, dtype), a.size)
    return c


def saxpy(dtype, alpha, x, y):
    """Return alpha*x + y (fused, binary32) as a new array; y is not modified."""
    x, y = _arr(x, dtype), _arr(y, dtype)
    if x.shape != y.shape:
        raise ValueError("shape mismatch")
    out = np.array(y, copy=True)
    getattr(lib(), "orc_saxpy_" + dtype)(ctypes.c_float(alpha), _ptr(x, dtype),
                                         _ptr(out, dtype), x.size)
    return out


def relu(dtype, x):
    """y = max(x, 0); x <= 0 (with -0) gives +0, NaN passes through."""
    x = _arr(x, dtype)
    y = np.empty_like(x)
    getattr(lib(), "orc_relu_" + dtype)(_ptr(x, dtype), _ptr(y, dtype), x.size)
    return y


def relu_inplace(dtype, x):
    """ReLU computed into the same array."""
    x = _arr(x, dtype)
    getattr(lib(), "orc_relu_" + dtype)(_ptr(x, dtype), _ptr(x, dtype), x.size)
    return x


def select_even_odd(x):
    """y = x even ? 2x : x + 1 on int32, wrapping modulo 2^32."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.int32:
        raise TypeError("select_even_odd expects int32, got %s" % x.dtype)
    y = np.empty_like(x)
    lib().orc_select_even_odd_i32(x.ctypes.data, y.ctypes.data, x.size)
    return y


def copy(x):
    """out[i] = in[i] (raw bits)."""
    x = np.ascontiguousarray(x)
    out = np.empty_like(x)
    lib().orc_copy(x.ctypes.data, out.ctypes.data, x.size, x.itemsize)
    return out


def gather_stride(x, s):
    """out[i] = in[(s*i) mod n] (raw bits)."""
    x = np.ascontiguousarray(x)
    out = np.empty_like(x)
    lib().orc_gather_stride(x.ctypes.data, out.ctypes.data, x.size, int(s), x.itemsize)
    return out


def gather_index(i, s, n):
    return lib().orc_gather_index(int(i), int(s), int(n))


def ceil_div(n, t):
    return lib().orc_ceil_div(int(n), int(t))


def f16_to_f64(h):
    return lib().orc_f16_to_f64(int(h))


def bf16_to_f64(h):
    return lib().orc_bf16_to_f64(int(h))


def f64_to_f16(x):
    return lib().orc_f64_to_f16(float(x))


def f64_to_bf16(x):
    return lib().orc_f64_to_bf16(float(x))


def decode_all(dtype):
    """Decode all 2^16 bit patterns of a 16-bit dtype to float64."""
    f = f16_to_f64 if dtype == "f16" else bf16_to_f64
    return np.array([f(h) for h in range(1 << 16)], dtype=np.float64)
