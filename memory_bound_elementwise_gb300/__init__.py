"""GB300-native memory-bound elementwise operators.

Thin Python binding over the C ABI of ``libew.so`` (declared in
``include/ew.h``): argument marshalling only.  Every operation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and calling an
operator without the built library raises.

Tensor entry points (same names as the C ABI)::

    ew_add(a, b, c=None)            C = A + B
    ew_saxpy(alpha, x, y)           y = alpha*x + y, in place
    ew_relu(x, y=None)              y = max(x, 0)  (y = x for in place)
    ew_add_relu(a, b, c=None)       C = max(A + B, 0), one pass
    ew_select_even_odd(x, y=None)   y = x even ? 2x : x + 1 (int32)
    ew_copy(x, out)                 out = x
    ew_gather_stride(x, out, s)     out[i] = x[(s*i) mod n]

Tensors must be contiguous CUDA tensors of dtype float32, float16 or bfloat16
(int32 for ew_select_even_odd, ew_copy and ew_gather_stride) on the current
device; calls are enqueued on ``stream`` (default: torch's
current stream) and do not synchronise.  ``lib()`` exposes the raw ctypes
handle with the exact C signatures.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libew.so")

# ew_dtype
EW_F32, EW_F16, EW_BF16, EW_I32 = 0, 1, 2, 3
# ew_path
PATH_AUTO, PATH_SCALAR, PATH_V128, PATH_V256, PATH_TMA = 0, 1, 2, 3, 4
PATH_NAMES = {PATH_AUTO: "auto", PATH_SCALAR: "scalar", PATH_V128: "v128",
              PATH_V256: "v256", PATH_TMA: "tma"}
# ew_schedule
SCHED_AUTO, SCHED_ONESHOT, SCHED_PERSISTENT, SCHED_LAPS, SCHED_TILED = 0, 1, 2, 3, 4
SCHED_NAMES = {SCHED_AUTO: "auto", SCHED_ONESHOT: "oneshot", SCHED_PERSISTENT: "persistent",
               SCHED_LAPS: "laps", SCHED_TILED: "tiled"}
# ew_status
EW_OK = 0
STATUS_NAMES = {0: "EW_OK", 1: "EW_ERR_INVALID_VALUE", 2: "EW_ERR_NULL_POINTER",
                3: "EW_ERR_UNSUPPORTED_DTYPE", 4: "EW_ERR_OVERLAP",
                5: "EW_ERR_NOT_DEVICE_POINTER", 6: "EW_ERR_CUDA", 7: "EW_ERR_TIMEOUT"}

# Every function declared in include/ew.h.
EXPORTS = ("ew_add", "ew_saxpy", "ew_relu", "ew_add_relu", "ew_saxpy_relu", "ew_select_even_odd", "ew_copy",
           "ew_gather_stride", "ew_set_path", "ew_set_programmatic_launch",
           "ew_get_programmatic_launch",
           "ew_get_path", "ew_set_schedule", "ew_get_schedule", "ew_set_pointer_check",
           "ew_plan_query", "ew_last_launch", "ew_gather_plan_query", "ew_status_string", "ew_last_cuda_error",
           "ew_device_error", "ew_selftest_bounded_wait", "ew_version")


class EwError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = "%s: %s" % (where, status_string(status))
        if status == 6:
            msg += " (cudaError_t %d)" % lib().ew_last_cuda_error()
        super().__init__(msg)


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("vec_bytes", ctypes.c_int32),
                ("head", ctypes.c_int64), ("nvec", ctypes.c_int64), ("tail", ctypes.c_int64)]


class LaunchRecord(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int32), ("path", ctypes.c_int32),
                ("vec_bytes", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("block", ctypes.c_int32), ("smem", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("head", ctypes.c_int64), ("nvec", ctypes.c_int64), ("tail", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_lib = None


def lib():
    """The loaded ``libew.so`` with argument types set; raises if not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libew.so is not built (%s). Build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`." % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    L.ew_add.argtypes = [ctypes.c_int, vp, vp, vp, i64, vp]
    L.ew_saxpy.argtypes = [ctypes.c_int, f32, vp, vp, i64, vp]
    L.ew_saxpy_relu.argtypes = [ctypes.c_int, f32, vp, vp, i64, vp]
    L.ew_relu.argtypes = [ctypes.c_int, vp, vp, i64, vp]
    L.ew_add_relu.argtypes = [ctypes.c_int, vp, vp, vp, i64, vp]
    L.ew_select_even_odd.argtypes = [ctypes.c_int, vp, vp, i64, vp]
    L.ew_copy.argtypes = [ctypes.c_int, vp, vp, i64, vp]
    L.ew_gather_stride.argtypes = [ctypes.c_int, vp, vp, i64, i64, vp]
    for name in ("ew_add", "ew_saxpy", "ew_relu", "ew_add_relu", "ew_saxpy_relu", "ew_select_even_odd", "ew_copy",
                 "ew_gather_stride",
                 "ew_set_path", "ew_set_schedule", "ew_set_pointer_check", "ew_plan_query",
                 "ew_last_launch", "ew_gather_plan_query", "ew_device_error", "ew_selftest_bounded_wait"):
        getattr(L, name).restype = ctypes.c_int
    L.ew_set_path.argtypes = [ctypes.c_int]
    L.ew_get_path.argtypes = []
    L.ew_get_path.restype = ctypes.c_int
    L.ew_set_schedule.argtypes = [ctypes.c_int]
    L.ew_get_schedule.argtypes = []
    L.ew_get_schedule.restype = ctypes.c_int
    L.ew_selftest_bounded_wait.argtypes = [i64, vp]
    L.ew_set_pointer_check.argtypes = [ctypes.c_int]
    L.ew_set_programmatic_launch.argtypes = [ctypes.c_int]
    L.ew_set_programmatic_launch.restype = ctypes.c_int
    L.ew_get_programmatic_launch.argtypes = []
    L.ew_get_programmatic_launch.restype = ctypes.c_int
    L.ew_plan_query.argtypes = [ctypes.c_int, ctypes.POINTER(vp), i32, i64, ctypes.POINTER(Plan)]
    L.ew_last_launch.argtypes = [ctypes.POINTER(LaunchRecord)]
    L.ew_gather_plan_query.argtypes = [ctypes.c_int, vp, vp, i64, i64, ctypes.POINTER(LaunchRecord)]
    L.ew_status_string.argtypes = [ctypes.c_int]
    L.ew_status_string.restype = ctypes.c_char_p
    L.ew_last_cuda_error.argtypes = []
    L.ew_last_cuda_error.restype = ctypes.c_int
    L.ew_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    L.ew_version.argtypes = []
    L.ew_version.restype = ctypes.c_int
    _lib = L
    return _lib


def status_string(status):
    return lib().ew_status_string(int(status)).decode()


def check(status, where):
    if status != EW_OK:
        raise EwError(status, where)


# ---------------------------------------------------------------- tensors

def _dtype_code(t):
    import torch
    codes = {torch.float32: EW_F32, torch.float16: EW_F16, torch.bfloat16: EW_BF16,
             torch.int32: EW_I32}
    if t.dtype not in codes:
        raise TypeError("unsupported dtype %s (float32, float16, bfloat16, int32)" % t.dtype)
    return codes[t.dtype]


def _check_tensors(*ts):
    t0 = ts[0]
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.dtype != t0.dtype or t.numel() != t0.numel() or t.device != t0.device:
            raise ValueError("tensors must share dtype, size and device")
    return _dtype_code(t0), t0.numel()


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def ew_add(a, b, c=None, stream=None):
    """C = A + B (c may be a or b for in place); returns c."""
    import torch
    if c is None:
        c = torch.empty_like(a)
    dt, n = _check_tensors(a, b, c)
    check(lib().ew_add(dt, a.data_ptr(), b.data_ptr(), c.data_ptr(), n, _stream(stream, a.device)),
          "ew_add")
    return c


def ew_saxpy(alpha, x, y, stream=None):
    """y = alpha * x + y in place (one fused multiply-add in binary32); returns y."""
    dt, n = _check_tensors(x, y)
    check(lib().ew_saxpy(dt, float(alpha), x.data_ptr(), y.data_ptr(), n, _stream(stream, x.device)),
          "ew_saxpy")
    return y


def ew_saxpy_relu(alpha, x, y, stream=None):
    """y = max(alpha * x + y, 0) in place, in one pass (the fma rounded first); returns y."""
    dt, n = _check_tensors(x, y)
    check(lib().ew_saxpy_relu(dt, float(alpha), x.data_ptr(), y.data_ptr(), n, _stream(stream, x.device)),
          "ew_saxpy_relu")
    return y


def ew_relu(x, y=None, stream=None):
    """y = max(x, 0) with -0 -> +0 and NaN kept; y = x computes in place."""
    import torch
    if y is None:
        y = torch.empty_like(x)
    dt, n = _check_tensors(x, y)
    check(lib().ew_relu(dt, x.data_ptr(), y.data_ptr(), n, _stream(stream, x.device)), "ew_relu")
    return y


def ew_add_relu(a, b, c=None, stream=None):
    """C = max(A + B, 0) in one pass (c may be a or b); returns c."""
    import torch
    if c is None:
        c = torch.empty_like(a)
    dt, n = _check_tensors(a, b, c)
    check(lib().ew_add_relu(dt, a.data_ptr(), b.data_ptr(), c.data_ptr(), n,
                            _stream(stream, a.device)), "ew_add_relu")
    return c


def ew_select_even_odd(x, y=None, stream=None):
    """y = x even ? 2x : x + 1 on int32 tensors (wrapping); y = x computes in place."""
    import torch
    if y is None:
        y = torch.empty_like(x)
    dt, n = _check_tensors(x, y)
    check(lib().ew_select_even_odd(dt, x.data_ptr(), y.data_ptr(), n, _stream(stream, x.device)),
          "ew_select_even_odd")
    return y


def ew_copy(x, out, stream=None):
    """out = x (raw bits); returns out."""
    dt, n = _check_tensors(x, out)
    check(lib().ew_copy(dt, x.data_ptr(), out.data_ptr(), n, _stream(stream, x.device)), "ew_copy")
    return out


def ew_gather_stride(x, out, stride, stream=None):
    """out[i] = x[(stride*i) mod n]; returns out."""
    dt, n = _check_tensors(x, out)
    check(lib().ew_gather_stride(dt, x.data_ptr(), out.data_ptr(), n, int(stride),
                                 _stream(stream, x.device)), "ew_gather_stride")
    return out


# ---------------------------------------------------------------- control

def set_path(path):
    """Select the kernel variant: 'auto', 'scalar', 'v128', 'v256' or 'tma'."""
    code = {v: k for k, v in PATH_NAMES.items()}[path] if isinstance(path, str) else int(path)
    check(lib().ew_set_path(code), "ew_set_path")


def get_path():
    return PATH_NAMES[lib().ew_get_path()]


def set_schedule(schedule):
    """Select the block schedule: 'auto', 'oneshot', 'persistent', 'laps' or
    'tiled' (the gather's lap order and its transposing tiles; the other
    operators run 'oneshot' under those two)."""
    code = ({v: k for k, v in SCHED_NAMES.items()}[schedule] if isinstance(schedule, str)
            else int(schedule))
    check(lib().ew_set_schedule(code), "ew_set_schedule")


def get_schedule():
    return SCHED_NAMES[lib().ew_get_schedule()]


def set_programmatic_launch(enable):
    """Programmatic dependent launch on (default) or off."""
    check(lib().ew_set_programmatic_launch(1 if enable else 0), "ew_set_programmatic_launch")


def get_programmatic_launch():
    return bool(lib().ew_get_programmatic_launch())


def set_pointer_check(enable):
    check(lib().ew_set_pointer_check(1 if enable else 0), "ew_set_pointer_check")


def plan_query(dtype_code, ptrs, n):
    """Host-side split of a call: dict(path, vec_bytes, head, nvec, tail)."""
    arr = (ctypes.c_void_p * len(ptrs))(*[ctypes.c_void_p(p) for p in ptrs])
    out = Plan()
    check(lib().ew_plan_query(dtype_code, arr, len(ptrs), int(n), ctypes.byref(out)), "ew_plan_query")
    return {k: getattr(out, k) for k, _ in Plan._fields_}


def gather_plan_query(dtype_code, in_ptr, out_ptr, n, stride):
    """The launch record an ew_gather_stride call would leave (host only; the
    grid-stride kernel's grid is 0), as last_launch() returns it."""
    rec = LaunchRecord()
    check(lib().ew_gather_plan_query(dtype_code, in_ptr, out_ptr, int(n), int(stride), ctypes.byref(rec)),
          "ew_gather_plan_query")
    return rec.as_dict()


def last_launch():
    rec = LaunchRecord()
    check(lib().ew_last_launch(ctypes.byref(rec)), "ew_last_launch")
    return rec.as_dict()


def selftest_bounded_wait(limit_ns, stream=None):
    """Enqueue the bounded-wait self-test (its wait must give up after limit_ns)."""
    import torch
    check(lib().ew_selftest_bounded_wait(int(limit_ns), _stream(stream, torch.cuda.current_device())),
          "ew_selftest_bounded_wait")


def device_error(stream=None):
    """Read and clear the device error word (one atomic exchange ordered on
    ``stream``), then synchronise ``stream``; returns (status, code)."""
    import torch
    code = ctypes.c_int32(0)
    st = lib().ew_device_error(_stream(stream, torch.cuda.current_device()), ctypes.byref(code))
    return st, code.value


__all__ = ["ew_add", "ew_saxpy", "ew_relu", "ew_add_relu", "ew_saxpy_relu", "ew_select_even_odd", "ew_copy",
           "ew_gather_stride", "set_path",
           "get_path", "set_schedule", "get_schedule", "set_programmatic_launch",
           "get_programmatic_launch", "set_pointer_check", "plan_query",
           "last_launch", "device_error", "selftest_bounded_wait", "lib", "EwError", "EXPORTS"]
