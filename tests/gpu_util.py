"""Helpers for the GPU parity tests: device buffers with guard zones, and
bit-level comparison against the oracle."""
import numpy as np
import torch

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "i32": torch.int32}
BITS_NP = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "i32": np.uint32}
BITS_T = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16, "i32": torch.int32}
ESIZE = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}
GUARD_BYTES = 4096
SENTINEL = 0x5A


class GuardedBuffer:
    """A device buffer of ``n`` elements starting ``offset`` elements past a
    256-byte boundary, with GUARD_BYTES of sentinel bytes on both sides."""

    def __init__(self, n, dtype, offset=0, device="cuda"):
        e = ESIZE[dtype]
        self.n, self.dtype, self.offset = n, dtype, offset
        self.lo = GUARD_BYTES + offset * e
        total = self.lo + n * e + GUARD_BYTES
        self.raw = torch.full((total,), SENTINEL, dtype=torch.uint8, device=device)
        assert self.raw.data_ptr() % 256 == 0
        self.view = self.raw[self.lo:self.lo + n * e].view(TORCH_DT[dtype])

    def fill(self, arr):
        b = np.ascontiguousarray(arr).view(np.uint8)
        self.raw[self.lo:self.lo + b.size].copy_(torch.from_numpy(b))
        return self

    def host(self):
        host_dt = {"f32": np.float32, "i32": np.int32}.get(self.dtype, np.uint16)
        return self.raw[self.lo:self.lo + self.n * ESIZE[self.dtype]].cpu().numpy().view(host_dt)

    def guards_intact(self):
        head = self.raw[:self.lo]
        tail = self.raw[self.lo + self.n * ESIZE[self.dtype]:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def is_nan_bits(bits, dtype):
    if dtype == "f32":
        return (bits & 0x7FFFFFFF) > 0x7F800000
    if dtype == "f16":
        return (bits & 0x7FFF) > 0x7C00
    return (bits & 0x7FFF) > 0x7F80


def assert_bits_equal(got, want, dtype, nan_as_class=False, what=""):
    """Bit-exact comparison; with ``nan_as_class`` any NaN matches any NaN
    (arithmetic results: the hardware returns a canonical NaN)."""
    g = np.ascontiguousarray(got).view(BITS_NP[dtype])
    w = np.ascontiguousarray(want).view(BITS_NP[dtype])
    assert g.shape == w.shape
    if nan_as_class:
        gn, wn = is_nan_bits(g, dtype), is_nan_bits(w, dtype)
        bad = np.nonzero((g != w) & ~(gn & wn))[0]
    else:
        bad = np.nonzero(g != w)[0]
    if bad.size:
        i = int(bad[0])
        raise AssertionError("%s: %d mismatches, first at %d: got %#x want %#x"
                             % (what, bad.size, i, int(g[i]), int(w[i])))
