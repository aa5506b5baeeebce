"""GPU parity: every operator, dtype and kernel variant against the oracle,
element by element, through the C ABI.

Small cases span several vectors, grid strides and ragged heads/tails at every
alignment offset; output buffers carry guard zones that must stay untouched.
The full-size cases are the measured workloads: fp32 add at 2^20+3 and 2^28,
fp32 SAXPY at 32M in place, bf16/fp16 add at 2^28 (aligned and offset by one
element), fp32 ReLU at 2^28 (out of place and in place), fp32 copy and
stride-2 gather at 2^26; and the bench's further workloads: bf16 add at
2^28 with pointers of different parity, fused SAXPY + ReLU at 2^28 and the
stride-16 gather at 2^26.
The bar is bit-exact; NaN results of arithmetic compare as "both NaN".
"""

import numpy as np
import pytest
import torch

import memory_bound_elementwise_gb300 as ew
import oracle
from memory_bound_elementwise_gb300 import inputs
from tests.gather_geometry import fixed_block
from tests.gpu_util import GuardedBuffer, assert_bits_equal, ESIZE

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]
PATHS = ["auto", "scalar", "v128", "v256", "tma"]
SMALL_N = [1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 64, 255, 257, 1000, 4099, 70001]
DT_CODE = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}


@pytest.fixture(autouse=True)
def _reset_path():
    ew.set_path("auto")
    ew.set_schedule("auto")
    yield
    ew.set_path("auto")
    ew.set_schedule("auto")
    assert ew.device_error() == (0, 0), "a bounded device wait gave up during the test"


def _stream():
    return torch.cuda.current_stream().cuda_stream


def run_op(op, dtype, bufs, n, alpha=2.5):
    """Call the C ABI directly with raw pointers."""
    L = ew.lib()
    dt = DT_CODE[dtype]
    p = [b.view.data_ptr() for b in bufs]
    if op == "add":
        st = L.ew_add(dt, p[0], p[1], p[2], n, _stream())
    elif op == "saxpy":
        st = L.ew_saxpy(dt, alpha, p[0], p[1], n, _stream())
    elif op == "relu":
        st = L.ew_relu(dt, p[0], p[1], n, _stream())
    elif op == "add_relu":
        st = L.ew_add_relu(dt, p[0], p[1], p[2], n, _stream())
    elif op == "saxpy_relu":
        st = L.ew_saxpy_relu(dt, alpha, p[0], p[1], n, _stream())
    elif op == "copy":
        st = L.ew_copy(dt, p[0], p[1], n, _stream())
    else:
        raise ValueError(op)
    assert st == 0, ew.status_string(st)


def expected(op, dtype, x, y, alpha=2.5):
    if op == "add":
        return oracle.add(dtype, x, y)
    if op == "saxpy":
        return oracle.saxpy(dtype, alpha, x, y)
    if op == "relu":
        return oracle.relu(dtype, x)
    if op == "add_relu":  # the unfused definition: round the sum, then ReLU
        return oracle.relu(dtype, oracle.add(dtype, x, y))
    if op == "saxpy_relu":  # round the fused multiply-add, then ReLU
        return oracle.relu(dtype, oracle.saxpy(dtype, alpha, x, y))
    return oracle.copy(x)


def make_inputs(dtype, n, seed, specials=True):
    x = inputs.as_dtype(inputs.normal(n, seed) * np.float32(3.0), dtype)
    y = inputs.as_dtype(inputs.uniform(n, seed + 1), dtype)
    if specials:
        x = inputs.with_specials(x, dtype, seed)
        y = inputs.with_specials(y, dtype, seed + 7)
    return x, y


def check_case(op, dtype, n, offs, seed, path="auto", schedule="auto"):
    x, y = make_inputs(dtype, n, seed)
    nin = {"add": 2, "add_relu": 2, "saxpy": 2, "saxpy_relu": 2, "relu": 1, "copy": 1}[op]
    if op in ("saxpy", "saxpy_relu"):
        bx = GuardedBuffer(n, dtype, offs[0]).fill(x)
        by = GuardedBuffer(n, dtype, offs[1]).fill(y)
        bufs, outb = [bx, by], by
    elif nin == 2:
        bx = GuardedBuffer(n, dtype, offs[0]).fill(x)
        by = GuardedBuffer(n, dtype, offs[1]).fill(y)
        bo = GuardedBuffer(n, dtype, offs[2])
        bufs, outb = [bx, by, bo], bo
    else:
        bx = GuardedBuffer(n, dtype, offs[0]).fill(x)
        bo = GuardedBuffer(n, dtype, offs[1])
        bufs, outb = [bx, bo], bo
    ew.set_path(path)
    ew.set_schedule(schedule)
    run_op(op, dtype, bufs, n)
    rec = ew.last_launch()
    torch.cuda.synchronize()
    want = expected(op, dtype, x, y)
    assert_bits_equal(outb.host(), want, dtype, nan_as_class=op in ("add", "saxpy", "add_relu", "saxpy_relu"),
                      what="%s %s n=%d offs=%s path=%s" % (op, dtype, n, offs, path))
    for b in bufs:
        assert b.guards_intact(), "guard zone written: %s %s n=%d offs=%s" % (op, dtype, n, offs)
    return rec


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["add", "saxpy", "relu", "copy", "add_relu", "saxpy_relu"])
def test_small_sizes_every_offset(op, dtype):
    per = 32 // ESIZE[dtype]
    for n in SMALL_N:
        for off in range(per):
            nin = 3 if op in ("add", "add_relu") else 2
            check_case(op, dtype, n, [off] * nin, seed=1000 + n * 37 + off)


@pytest.mark.parametrize("schedule", ["oneshot", "persistent", "laps"])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["add", "saxpy", "relu", "copy", "add_relu", "saxpy_relu"])
def test_forced_paths(op, dtype, path, schedule):
    for n in (1, 33, 1000, 70001, 600_001):
        for off in (0, 1, 3):
            nin = 3 if op in ("add", "add_relu") else 2
            rec = check_case(op, dtype, n, [off] * nin, seed=2000 + n + off, path=path,
                             schedule=schedule)
            if path == "scalar":
                assert rec["vec_bytes"] == ESIZE[dtype]
            elif path == "v128":
                assert rec["vec_bytes"] <= 16
            elif path == "tma":
                assert rec["path"] == 4 and rec["vec_bytes"] == 16
            if path != "tma" and rec["nvec"] > 0:
                # lap order exists for the gather only: the streaming kernels run one-shot
                assert rec["schedule"] == (2 if schedule == "persistent" else 1)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["add", "saxpy", "relu", "copy", "add_relu", "saxpy_relu"])
def test_tma_tile_boundaries(op, dtype):
    """Sizes around the 8 KiB bulk-copy tile and the 2-tile CTA, at offsets that
    keep or break 16-byte alignment (the latter falls back to vector loads)."""
    per_tile = 8192 // ESIZE[dtype]
    sizes = [1, per_tile - 1, per_tile, per_tile + 1, 2 * per_tile, 2 * per_tile + 5,
             3 * per_tile + 7, 5 * per_tile - 3, 70001]
    for n in sizes:
        for off in (0, 1, 16 // ESIZE[dtype], 3):
            nin = 3 if op in ("add", "add_relu") else 2
            rec = check_case(op, dtype, n, [off] * nin, seed=2500 + n + off, path="tma")
            assert rec["path"] == 4
            assert rec["head"] + rec["nvec"] * per_tile + rec["tail"] == n


REALIGN_OFFSETS = {2: [[1, 0, 3], [0, 1, 0], [1, 1, 0], [3, 6, 7], [7, 0, 5], [0, 0, 1], [2, 5, 0], [0, 8, 3]],
                   4: [[1, 0, 3], [0, 1, 0], [3, 2, 1], [0, 0, 1], [2, 0, 2]]}


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", ["add", "saxpy", "relu", "copy", "add_relu", "saxpy_relu"])
def test_tma_realign_mixed_offsets(op, dtype):
    """EW_PATH_TMA with pointers that disagree modulo 16 bytes runs the
    realigning bulk-copy kernel: 16-byte aligned output tiles, each input
    staged as the aligned span around its tile and read at its offset.  Every
    input shift (2-byte steps for 16-bit types), sizes around one and several
    tiles and around the 16-byte margins kept at both ends."""
    e = ESIZE[dtype]
    per_tile = 8192 // e
    m = 16 // e
    sizes = [1, m, 2 * m, 3 * m + per_tile - 1, 3 * m + per_tile, 3 * m + per_tile + 1,
             3 * per_tile + 7, 70001]
    nin = 3 if op in ("add", "add_relu") else 2
    for n in sizes:
        for offs in REALIGN_OFFSETS[e]:
            offs = offs[:nin]
            rec = check_case(op, dtype, n, offs, seed=2700 + n + 7 * sum(offs), path="tma")
            assert rec["path"] == 4
            assert rec["head"] + rec["nvec"] * per_tile + rec["tail"] == n
            if len({(o * e) % 16 for o in offs}) > 1:  # offsets disagree modulo 16 bytes
                staged = 2 if op in ("add", "add_relu", "saxpy", "saxpy_relu") else 1  # inputs staged per tile
                assert rec["smem"] == 2 * (staged * (8192 + 16) + 8192) + 16, rec
                assert rec["head"] * e >= 16 or rec["nvec"] == 0
                assert rec["nvec"] == 0 or rec["tail"] * e >= 16


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", ["add", "saxpy", "relu", "copy", "add_relu", "saxpy_relu"])
def test_auto_realigns_16bit_parity_mismatch(op, dtype):
    """Under EW_PATH_AUTO, 16-bit pointers of different parity take the
    realigning bulk-copy kernel from n = 2^22 (2-byte accesses below)."""
    nin = 3 if op in ("add", "add_relu") else 2
    for n, offs in (((1 << 22) + 4099, [1, 0, 3]), ((1 << 22) + 1, [0, 1, 0]), ((1 << 22) - 1, [1, 0, 3]),
                    ((1 << 22) + 7, [3, 6, 7])):
        rec = check_case(op, dtype, n, offs[:nin], seed=2900 + n + sum(offs))
        mismatch = len({o % 2 for o in offs[:nin]}) > 1
        if n >= 1 << 22 and mismatch:
            assert rec["path"] == 4 and rec["head"] + rec["nvec"] * 4096 + rec["tail"] == n, rec
        else:
            assert rec["path"] != 4, rec


def test_auto_realign_keeps_host_memory_on_vector_kernels():
    """AUTO sends only device memory to the realigning bulk copy: the same
    mixed-parity bf16 add on page-locked host buffers runs the vector kernel
    over the CPU-GPU link, and still matches the oracle."""
    n = (1 << 22) + 5
    x, y = make_inputs("bf16", n + 8, 3300)
    hx = torch.from_numpy(x.view(np.int16)).pin_memory()
    hy = torch.from_numpy(y.view(np.int16)).pin_memory()
    hz = torch.zeros(n + 8, dtype=torch.int16).pin_memory()
    assert ew.lib().ew_add(2, hx.data_ptr() + 2, hy.data_ptr(), hz.data_ptr() + 6, n, _stream()) == 0
    rec = ew.last_launch()
    assert rec["path"] != 4 and rec["vec_bytes"] == 2, rec
    torch.cuda.synchronize()
    got = hz.numpy().view(np.uint16)[3:3 + n]
    assert_bits_equal(got, oracle.add("bf16", x[1:1 + n], y[:n]), "bf16", True, "host mixed parity")
    # device copies of the same arrays take the realigning kernel
    dx, dy, dz = hx.cuda(), hy.cuda(), hz.cuda()
    assert ew.lib().ew_add(2, dx.data_ptr() + 2, dy.data_ptr(), dz.data_ptr() + 6, n, _stream()) == 0
    assert ew.last_launch()["path"] == 4
    torch.cuda.synchronize()
    assert_bits_equal(dz.cpu().numpy().view(np.uint16)[3:3 + n], got, "bf16", True, "device mixed parity")


def test_bounded_wait_gives_up_and_reports():
    """The self-test block arms an mbarrier that nothing completes: its wait
    must end after the limit with code 99, and the word must read clear after."""
    import time
    t0 = time.perf_counter()
    ew.selftest_bounded_wait(50_000_000)  # 50 ms
    st, code = ew.device_error()
    elapsed = time.perf_counter() - t0
    assert (st, code) == (7, 99)
    assert 0.04 < elapsed < 5.0
    assert ew.device_error() == (0, 0)
    # the context is still usable afterwards
    x = torch.arange(1000, dtype=torch.float32, device="cuda")
    y = ew.ew_relu(x - 500)
    torch.cuda.synchronize()
    assert float(y.sum()) == float(sum(range(1, 500)))


def test_device_error_read_on_another_stream():
    """The error word is taken out by an atomic exchange ordered on the
    reading stream: a code recorded by a kernel on stream A is returned by a
    read on stream B once A's work is done, exactly once."""
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    assert ew.device_error() == (0, 0)
    ew.selftest_bounded_wait(20_000_000, stream=a)  # 20 ms
    a.synchronize()
    assert ew.device_error(stream=b) == (7, 99)
    assert ew.device_error(stream=a) == (0, 0)
    assert ew.device_error(stream=b) == (0, 0)


LAP_BLOCK = 2048  # outputs per block of the lap-ordered gather (256 threads x 8)


def _gather_laps(n, s):
    """Whether ew_gather_stride takes the lap-ordered kernel under schedule 'laps'."""
    sm = s % n
    return 2 <= sm <= 64 and n <= 1 << 32 and n // sm >= LAP_BLOCK


def _gather_auto_schedule(n, s, dtype):
    """The schedule AUTO picks: tiled up to s = 64, from s = 5 for 4-byte
    elements and from s = 2 for 2-byte ones; lap order below that where
    every lap holds a block, else index order."""
    sm = s % n
    if n > 1 << 32:
        return 2
    if (5 if ESIZE[dtype] == 4 else 2) <= sm <= 64:
        return 4
    return 3 if _gather_laps(n, s) else 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gather_schedules_agree(dtype):
    L = ew.lib()
    for sched in ("oneshot", "persistent", "laps", "auto"):
        ew.set_schedule(sched)
        for n in (1, 5, 4097, 300_001):
            x = inputs.random_bits(n, dtype, 6500 + n)
            for s in (2, 3, n + 1, (1 << 33) + 1):
                bi = GuardedBuffer(n, dtype, 1).fill(x)
                bo = GuardedBuffer(n, dtype, 0)
                assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(),
                                          n, s, _stream()) == 0
                rec = ew.last_launch()
                if sched == "persistent":
                    assert rec["schedule"] == 2
                elif sched == "auto":
                    assert rec["schedule"] == _gather_auto_schedule(n, s, dtype), (n, s, rec)
                elif sched == "oneshot" or not _gather_laps(n, s):
                    assert rec["schedule"] == 1
                else:
                    assert rec["schedule"] == 3
                torch.cuda.synchronize()
                assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False,
                                  "gather %s n=%d s=%d" % (sched, n, s))
                assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("dtype", DTYPES)
def test_mixed_offsets_fall_back(dtype):
    for offs in ([1, 0, 3], [0, 2, 4], [4, 0, 8], [2, 6, 10], [0, 0, 1], [5, 5, 13],
                 [0, 1, 0], [1, 1, 0], [1, 0, 0], [0, 1, 1]):
        for n in (1, 2, 3, 4, 5, 6, 7, 17, 1000, 4099, 70001):
            check_case("add", dtype, n, offs, seed=3000 + n + sum(offs))
            check_case("saxpy", dtype, n, offs[:2], seed=3100 + n + sum(offs))
            check_case("relu", dtype, n, offs[:2], seed=3200 + n + sum(offs))


@pytest.mark.parametrize("dtype", DTYPES)
def test_saxpy_special_alphas(dtype):
    """alpha = +-0, +-inf, NaN, a subnormal, the largest binary32, 1/3: the
    fused multiply-add must match the oracle for every input class."""
    n = 4099
    L = ew.lib()
    alphas = [0.0, -0.0, float("inf"), float("-inf"), float("nan"),
              float(np.float32(1e-40)), float(np.finfo(np.float32).max), float(np.float32(1 / 3))]
    for k, alpha in enumerate(alphas):
        x, y = make_inputs(dtype, n, 4600 + k)
        bx = GuardedBuffer(n, dtype, 1).fill(x)
        by = GuardedBuffer(n, dtype, 1).fill(y)
        assert L.ew_saxpy(DT_CODE[dtype], alpha, bx.view.data_ptr(), by.view.data_ptr(), n, _stream()) == 0
        torch.cuda.synchronize()
        assert_bits_equal(by.host(), oracle.saxpy(dtype, alpha, x, y), dtype, True,
                          "saxpy alpha=%r" % alpha)
        assert by.guards_intact()


@pytest.mark.parametrize("dtype", DTYPES)
def test_saxpy_relu_special_alphas_and_aliasing(dtype):
    """Fused SAXPY + ReLU: alpha = +-0, +-inf, NaN, a subnormal, the largest
    binary32 and 1/3 against the oracle's saxpy then relu; x == y in place;
    and a 2^24-element case spanning many blocks."""
    L = ew.lib()
    n = 4099
    alphas = [0.0, -0.0, float("inf"), float("-inf"), float("nan"),
              float(np.float32(1e-40)), float(np.finfo(np.float32).max), float(np.float32(1 / 3))]
    for k, alpha in enumerate(alphas):
        x, y = make_inputs(dtype, n, 4700 + k)
        bx = GuardedBuffer(n, dtype, 1).fill(x)
        by = GuardedBuffer(n, dtype, 1).fill(y)
        assert L.ew_saxpy_relu(DT_CODE[dtype], alpha, bx.view.data_ptr(), by.view.data_ptr(), n,
                               _stream()) == 0
        torch.cuda.synchronize()
        want = oracle.relu(dtype, oracle.saxpy(dtype, alpha, x, y))
        assert_bits_equal(by.host(), want, dtype, True, "saxpy_relu alpha=%r" % alpha)
        assert by.guards_intact()
    x, _ = make_inputs(dtype, n, 4750)
    bx = GuardedBuffer(n, dtype, 0).fill(x)
    assert L.ew_saxpy_relu(DT_CODE[dtype], -1.5, bx.view.data_ptr(), bx.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(bx.host(), oracle.relu(dtype, oracle.saxpy(dtype, -1.5, x, x)), dtype, True,
                      "saxpy_relu x == y")
    m = 1 << 24
    x = inputs.as_dtype(inputs.normal(m, 4760), dtype)
    y = inputs.as_dtype(inputs.normal(m, 4761), dtype)
    tx = torch.from_numpy(x.view(np.int32 if dtype == "f32" else np.int16)).cuda()
    ty = torch.from_numpy(y.view(np.int32 if dtype == "f32" else np.int16)).cuda()
    assert L.ew_saxpy_relu(DT_CODE[dtype], 2.5, tx.data_ptr(), ty.data_ptr(), m, _stream()) == 0
    torch.cuda.synchronize()
    got = ty.cpu().numpy().view(np.float32 if dtype == "f32" else np.uint16)
    assert_bits_equal(got, oracle.relu(dtype, oracle.saxpy(dtype, 2.5, x, y)), dtype, True, "saxpy_relu 2^24")


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(dtype):
    n = 70001
    x, y = make_inputs(dtype, n, 4000)
    L = ew.lib()
    dt = DT_CODE[dtype]
    # c == a
    ba = GuardedBuffer(n, dtype, 1).fill(x)
    bb = GuardedBuffer(n, dtype, 1).fill(y)
    assert L.ew_add(dt, ba.view.data_ptr(), bb.view.data_ptr(), ba.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(ba.host(), oracle.add(dtype, x, y), dtype, True, "add in place")
    # saxpy with x == y
    bx = GuardedBuffer(n, dtype, 0).fill(x)
    assert L.ew_saxpy(dt, -0.75, bx.view.data_ptr(), bx.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(bx.host(), oracle.saxpy(dtype, -0.75, x, x), dtype, True, "saxpy x==y")
    # relu in place
    br = GuardedBuffer(n, dtype, 3).fill(x)
    assert L.ew_relu(dt, br.view.data_ptr(), br.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(br.host(), oracle.relu(dtype, x), dtype, False, "relu in place")
    for b in (ba, bb, bx, br):
        assert b.guards_intact()


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place_relu_skips_unchanged_vectors(dtype):
    """In place, vectors ReLU leaves unchanged are not stored; results must be
    the same as computing every element, including on a second pass where
    nothing changes and on inputs that are mostly non-negative."""
    n = 300_007
    L = ew.lib()
    x = inputs.as_dtype(inputs.normal(n, 4500), dtype)
    mostly_pos = inputs.as_dtype(np.abs(inputs.normal(n, 4501)), dtype)
    mostly_pos[::997] = inputs.as_dtype(np.float32([-1.0]), dtype)[0]  # a few negatives
    for src in (x, mostly_pos):
        for off in (0, 1, 3):
            b = GuardedBuffer(n, dtype, off).fill(src)
            want = oracle.relu(dtype, src)
            for _ in range(2):
                assert L.ew_relu(DT_CODE[dtype], b.view.data_ptr(), b.view.data_ptr(), n, _stream()) == 0
                torch.cuda.synchronize()
                assert_bits_equal(b.host(), want, dtype, False, "relu in place off=%d" % off)
            assert b.guards_intact()


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_bit_pattern_add_relu(dtype):
    """All 16-bit patterns (or 2^20 random binary32 patterns) as inputs."""
    if dtype == "f32":
        x = inputs.random_bits(1 << 20, "f32", 5000)
        y = inputs.random_bits(1 << 20, "f32", 5001)
    else:
        allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        x = np.tile(allp, 64)
        y = inputs.random_bits(x.size, dtype, 5002)
    n = x.size
    bx = GuardedBuffer(n, dtype).fill(x)
    by = GuardedBuffer(n, dtype).fill(y)
    bo = GuardedBuffer(n, dtype)
    run_op("add", dtype, [bx, by, bo], n)
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.add(dtype, x, y), dtype, True, "add all patterns")
    run_op("relu", dtype, [bx, bo], n)
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.relu(dtype, x), dtype, False, "relu all patterns")
    run_op("add_relu", dtype, [bx, by, bo], n)
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.relu(dtype, oracle.add(dtype, x, y)), dtype, True,
                      "add_relu all patterns")
    by.fill(y)
    run_op("saxpy", dtype, [bx, by], n, alpha=-1.5)
    torch.cuda.synchronize()
    assert_bits_equal(by.host(), oracle.saxpy(dtype, -1.5, x, y), dtype, True, "saxpy all patterns")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_add_16bit_every_pattern_against_4096_partners(dtype):
    """2^28 operand pairs per 16-bit format: every bit pattern as A against
    4096 seeded patterns as B (specials included), packed add on the GPU
    against the oracle's correctly rounded sum."""
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    partners = inputs.random_bits(4096, dtype, 8800)
    partners[:inputs.SPECIAL_BITS[dtype].size] = inputs.SPECIAL_BITS[dtype]
    x = np.tile(allp, partners.size)
    y = np.repeat(partners, allp.size)
    n = x.size
    bx = GuardedBuffer(n, dtype).fill(x)
    by = GuardedBuffer(n, dtype).fill(y)
    bo = GuardedBuffer(n, dtype)
    run_op("add", dtype, [bx, by, bo], n)
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.add(dtype, x, y), dtype, True, "add 2^28 pairs")
    assert bo.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_gather_small(dtype):
    L = ew.lib()
    for n in (1, 2, 3, 8, 33, 1000, 4097, 70001, 262144):
        x = inputs.random_bits(n, dtype, 6000 + n)
        for s in (1, 2, 3, 7, n + 2, (1 << 40) + 3):
            bi = GuardedBuffer(n, dtype, 1).fill(x)
            bo = GuardedBuffer(n, dtype, 0)
            assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(),
                                      n, s, _stream()) == 0
            torch.cuda.synchronize()
            assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False,
                              "gather n=%d s=%d" % (n, s))
            assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_gather_lap_order(dtype):
    """The lap-ordered gather (schedule 'laps'; AUTO's choice below s = 5)
    for strides 2..64 once every lap holds a block of outputs: sizes at, just below and just above the
    threshold n = 2048 s, laps of unequal length (s not dividing n), laps that
    read the same sources (s | n) and laps on distinct residues (s coprime to
    n), stride 65 and strides above n, misaligned input and output."""
    L = ew.lib()
    ew.set_schedule("laps")
    cases = []
    for s in (2, 3, 4, 5, 7, 8, 16, 31, 33, 64, 65):
        for n in (LAP_BLOCK * s - 1, LAP_BLOCK * s, LAP_BLOCK * s + 1, 3 * LAP_BLOCK * s + 5, 200_003):
            cases.append((n, s))
    cases += [(1 << 20, (1 << 20) + 2), (1 << 20, 3 * (1 << 20) + 5), (1 << 20, 2 + (1 << 40) * (1 << 20))]
    for n, s in cases:
        x = inputs.random_bits(n, dtype, 6700 + n + s)
        bi = GuardedBuffer(n, dtype, 3).fill(x)
        bo = GuardedBuffer(n, dtype, 1)
        assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(),
                                  n, s, _stream()) == 0
        rec = ew.last_launch()
        laps = _gather_laps(n, s)
        assert rec["schedule"] == (3 if laps else 1), (n, s, rec)
        if laps:
            sm = s % n
            lap_len = -(-n // sm)
            assert rec["grid"] == sm * -(-lap_len // LAP_BLOCK), (n, s, rec)
        torch.cuda.synchronize()
        assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False,
                          "lap gather n=%d s=%d" % (n, s))
        assert bi.guards_intact() and bo.guards_intact()


def test_launch_record_and_grid():
    n = 1 << 22
    a = torch.zeros(n, device="cuda")
    b = torch.zeros(n, device="cuda")
    ew.ew_add(a, b, torch.empty_like(a))
    rec = ew.last_launch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert rec["launches"] == 1 and rec["vec_bytes"] == 32 and rec["path"] == 3
    assert 1 <= rec["grid"] <= sms * (2048 // rec["block"])
    assert rec["nvec"] == n // 8 and rec["head"] == 0 and rec["tail"] == 0
    torch.cuda.synchronize()


def test_pointer_check_and_host_resident_buffers():
    """With the pointer check on, pageable host memory is accepted exactly when
    the device can access it (pageable memory access), and then computed over
    the CPU-GPU link like device memory; page-locked host memory always is."""
    n = 100_003
    a, b = inputs.uniform(n, 7100), inputs.uniform(n, 7101)
    want = oracle.add("f32", a, b)
    ew.set_pointer_check(True)
    try:
        # pageable host memory (numpy arrays): reachable on coherent CPU-GPU
        # systems such as GB300, rejected elsewhere
        c = np.empty_like(a)
        st = ew.lib().ew_add(0, a.ctypes.data, b.ctypes.data, c.ctypes.data, n, _stream())
        assert st in (0, 5)
        if st == 0:
            torch.cuda.synchronize()
            assert_bits_equal(c, want, "f32", True, "pageable host buffers")
        # page-locked host memory
        ta, tb = torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()
        tc = torch.empty(n).pin_memory()
        assert ew.lib().ew_add(0, ta.data_ptr(), tb.data_ptr(), tc.data_ptr(), n, _stream()) == 0
        torch.cuda.synchronize()
        assert_bits_equal(tc.numpy(), want, "f32", True, "pinned host buffers")
        # mixed: host inputs, device output
        d = torch.empty(n, device="cuda")
        assert ew.lib().ew_add(0, ta.data_ptr(), tb.data_ptr(), d.data_ptr(), n, _stream()) == 0
        torch.cuda.synchronize()
        assert_bits_equal(d.cpu().numpy(), want, "f32", True, "host inputs, device output")
    finally:
        ew.set_pointer_check(False)
    torch.cuda.synchronize()



def test_device_error_word_starts_clear():
    st, code = ew.device_error()
    assert (st, code) == (0, 0)


def test_binding_tensor_api_matches_oracle():
    n = 4099
    x, y = make_inputs("bf16", n, 7000, specials=False)
    tx = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    ty = torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16)
    tc = ew.ew_add(tx, ty)
    got = tc.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_bits_equal(got, oracle.add("bf16", x, y), "bf16", True, "binding add")
    with pytest.raises(ValueError):
        ew.ew_add(tx, ty[:-1])
    with pytest.raises(TypeError):
        ew.ew_relu(tx.to(torch.float64))


# ------------------------------------------------------------ full-size configs


def _full(op, dtype, n, seed_x, seed_y, offset=0, dist="uniform", inplace=False, alpha=2.5):
    if dist == "uniform":
        x = inputs.as_dtype(inputs.uniform(n, seed_x), dtype)
        y = inputs.as_dtype(inputs.uniform(n, seed_y), dtype)
    else:
        x = inputs.as_dtype(inputs.normal(n, seed_x), dtype)
        y = inputs.as_dtype(inputs.normal(n, seed_y), dtype) if op in ("add", "saxpy") else None
    if op == "relu":
        x = inputs.normal(n, seed_x)
        inputs.inject_signed_zeros(x)
        x = inputs.as_dtype(x, dtype)
    bx = GuardedBuffer(n, dtype, offset).fill(x)
    if op == "add":
        by = GuardedBuffer(n, dtype, offset).fill(y)
        bo = GuardedBuffer(n, dtype, offset)
        run_op("add", dtype, [bx, by, bo], n)
        want = oracle.add(dtype, x, y)
    elif op == "saxpy":
        by = GuardedBuffer(n, dtype, offset).fill(y)
        bo = by
        run_op("saxpy", dtype, [bx, by], n, alpha=alpha)
        want = oracle.saxpy(dtype, alpha, x, y)
    elif op == "relu":
        bo = bx if inplace else GuardedBuffer(n, dtype, offset)
        run_op("relu", dtype, [bx, bo], n)
        want = oracle.relu(dtype, x)
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), want, dtype, op != "relu", "%s %s n=%d" % (op, dtype, n))
    assert bo.guards_intact()
    return ew.last_launch()


def test_config_add_f32_odd_tail():
    rec = _full("add", "f32", (1 << 20) + 3, inputs.seed_for("add_f32_small"),
                inputs.seed_for("add_f32_small", 1))
    assert rec["tail"] == 3


def test_config_saxpy_f32_32M_in_place():
    _full("saxpy", "f32", 32 << 20, inputs.seed_for("saxpy_f32"), inputs.seed_for("saxpy_f32", 1),
          dist="normal")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_config_add_16bit_2p28(dtype, offset):
    rec = _full("add", dtype, 1 << 28, inputs.seed_for("add_16"), inputs.seed_for("add_16", 1),
                offset=offset, dist="normal")
    assert rec["head"] == (15 if offset else 0)


def test_bf16_add_2p28_pointers_of_different_parity():
    """The bench's mixed-parity workload at full size: bf16 add of 2^28
    elements with A, B and C at +1, +0 and +3 elements, which AUTO sends to the
    realigning bulk copy; every output against the oracle."""
    n = 1 << 28
    x = inputs.as_dtype(inputs.normal(n, inputs.seed_for("add_16")), "bf16")
    y = inputs.as_dtype(inputs.normal(n, inputs.seed_for("add_16", 1)), "bf16")
    ba, bb, bc = GuardedBuffer(n, "bf16", 1).fill(x), GuardedBuffer(n, "bf16", 0).fill(y), GuardedBuffer(n, "bf16", 3)
    run_op("add", "bf16", [ba, bb, bc], n)
    rec = ew.last_launch()
    assert rec["path"] == 4 and rec["head"] + rec["nvec"] * 4096 + rec["tail"] == n, rec
    torch.cuda.synchronize()
    assert_bits_equal(bc.host(), oracle.add("bf16", x, y), "bf16", True, "bf16 add 2^28 mixed parity")
    assert ba.guards_intact() and bb.guards_intact() and bc.guards_intact()


def test_saxpy_relu_f32_2p28():
    """The bench's fused SAXPY + ReLU workload at full size (alpha = 2.5)."""
    n = 1 << 28
    x = inputs.normal(n, inputs.seed_for("saxpy_f32", 2))
    y = inputs.normal(n, inputs.seed_for("saxpy_f32", 3))
    bx, by = GuardedBuffer(n, "f32").fill(x), GuardedBuffer(n, "f32").fill(y)
    run_op("saxpy_relu", "f32", [bx, by], n)
    torch.cuda.synchronize()
    assert_bits_equal(by.host(), oracle.relu("f32", oracle.saxpy("f32", 2.5, x, y)), "f32", True,
                      "saxpy_relu 2^28")
    assert by.guards_intact()


def test_gather_stride16_f32_2p26():
    """The bench's stride-16 gather at full size, through AUTO's tiled kernel."""
    n = 1 << 26
    x = inputs.uniform(n, inputs.seed_for("copy_f32"), 0.0, 1.0)
    bi, bo = GuardedBuffer(n, "f32").fill(x), GuardedBuffer(n, "f32")
    assert ew.lib().ew_gather_stride(0, bi.view.data_ptr(), bo.view.data_ptr(), n, 16, _stream()) == 0
    assert ew.last_launch()["schedule"] == 4
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.gather_stride(x, 16), "f32", False, "gather 16 2^26")
    assert bo.guards_intact() and bi.guards_intact()


@pytest.mark.parametrize("inplace", [False, True])
def test_config_relu_f32_2p28(inplace):
    _full("relu", "f32", 1 << 28, inputs.seed_for("relu_f32"), None, inplace=inplace)


def test_config_copy_and_gather_f32_2p26():
    n = 1 << 26
    x = inputs.uniform(n, inputs.seed_for("copy_f32"), 0.0, 1.0)
    bi = GuardedBuffer(n, "f32").fill(x)
    bo = GuardedBuffer(n, "f32")
    assert ew.lib().ew_copy(0, bi.view.data_ptr(), bo.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), x, "f32", False, "copy 2^26")
    assert ew.lib().ew_gather_stride(0, bi.view.data_ptr(), bo.view.data_ptr(), n, 2, _stream()) == 0
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.gather_stride(x, 2), "f32", False, "gather 2^26")
    assert bo.guards_intact() and bi.guards_intact()


def test_add_relu_f32_2p26():
    n = 1 << 26
    a = inputs.normal(n, inputs.seed_for("add_f32"))
    b = inputs.normal(n, inputs.seed_for("add_f32", 1))
    ba, bb, bc = GuardedBuffer(n, "f32").fill(a), GuardedBuffer(n, "f32").fill(b), GuardedBuffer(n, "f32")
    run_op("add_relu", "f32", [ba, bb, bc], n)
    torch.cuda.synchronize()
    assert_bits_equal(bc.host(), oracle.relu("f32", oracle.add("f32", a, b)), "f32", True, "add_relu 2^26")
    assert bc.guards_intact()


def test_config_add_f32_2p28():
    _full("add", "f32", 1 << 28, inputs.seed_for("add_f32"), inputs.seed_for("add_f32", 1))


@pytest.mark.parametrize("path,schedule", [("tma", "auto"), ("v256", "persistent")])
def test_config_add_f32_2p28_other_variants(path, schedule):
    """The headline workload through the bulk-copy path and the persistent schedule."""
    ew.set_path(path)
    ew.set_schedule(schedule)
    rec = _full("add", "f32", 1 << 28, inputs.seed_for("add_f32"), inputs.seed_for("add_f32", 1))
    assert rec["path"] == (4 if path == "tma" else 3)


def test_beyond_2p31_elements_f16():
    """n > 2^31 (byte offsets past 2^32): a seeded 2^20-element tile repeated on
    the device; every output tile and the ragged end compared with the oracle."""
    tile = 1 << 20
    n = (1 << 31) + 17
    a = inputs.as_dtype(inputs.normal(tile, 8100), "f16")
    b = inputs.as_dtype(inputs.normal(tile, 8101), "f16")
    reps = -(-n // tile)
    ta = torch.from_numpy(a.view(np.int16)).cuda().repeat(reps)[:n].contiguous()
    tb = torch.from_numpy(b.view(np.int16)).cuda().repeat(reps)[:n].contiguous()
    tc = torch.empty_like(ta)
    assert ew.lib().ew_add(1, ta.data_ptr(), tb.data_ptr(), tc.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    want = torch.from_numpy(oracle.add("f16", a, b).view(np.int16)).cuda()
    full = (n // tile) * tile
    assert torch.equal(tc[:full].view(-1, tile), want.expand(n // tile, tile))
    assert torch.equal(tc[full:], want[:n - full])
    del ta, tb, tc
    torch.cuda.empty_cache()


def test_gather_beyond_2p32_elements_f16():
    """n > 2^32 switches the gather to the grid-stride kernel (the one-shot
    index needs s*i < 2^64): input is a seeded 2^20-element tile repeated on the
    device; 200k sampled outputs and both ends are checked against the oracle's
    index map and the tile."""
    tile_n = 1 << 20
    n = (1 << 32) + 5
    s = 3
    tile = inputs.random_bits(tile_n, "f16", 8200)
    reps = -(-n // tile_n)
    tin = torch.from_numpy(tile.view(np.int16)).cuda().repeat(reps)[:n].contiguous()
    tout = torch.empty_like(tin)
    assert ew.lib().ew_gather_stride(1, tin.data_ptr(), tout.data_ptr(), n, s, _stream()) == 0
    rec = ew.last_launch()
    assert rec["schedule"] == 2  # grid-stride kernel above 2^32 elements
    torch.cuda.synchronize()
    g = inputs.rng(8201)
    idx = np.concatenate([np.arange(0, 1000), np.arange(n - 1000, n),
                          g.integers(0, n, size=200_000, dtype=np.int64)])
    got = tout[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint16)
    src = np.array([oracle.gather_index(int(i), s, n) for i in idx], dtype=np.int64)
    want = tile[src % tile_n]
    assert np.array_equal(got, want)
    del tin, tout
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_gather_tiled(dtype):
    """The tiled (transposing) gather for strides 2..64: strides that divide n
    (laps share one residue row), that are coprime to n (every row used once),
    even strides whose padded rows still share banks, ragged last blocks and
    n just above s.  Stride 65 and strides above n fall back to index order."""
    L = ew.lib()
    ew.set_schedule("tiled")
    for s in (2, 3, 4, 5, 6, 7, 8, 12, 16, 31, 33, 64, 65, (1 << 40) + 6):
        for n, in_off in ((s % (1 << 20) + 1, 0), (1000, 1), (8191, 0), (70001, 1), (300_007, 0),
                          (1 << 18, 1), ((1 << 18) + 3, 0)):
            x = inputs.random_bits(n, dtype, 7100 + n + s % 1000)
            bi = GuardedBuffer(n, dtype, in_off).fill(x)  # offset 0: 16-byte loads
            bo = GuardedBuffer(n, dtype, 3)
            assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(),
                                      n, s, _stream()) == 0
            rec = ew.last_launch()
            assert rec["schedule"] == (4 if 2 <= s % n <= 64 else 1), (n, s, rec)
            torch.cuda.synchronize()
            assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False,
                              "tiled gather n=%d s=%d" % (n, s))
            assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gather_tiled_general_every_input_offset(dtype):
    """Tiled gathers on every input offset within 16 bytes: the general
    kernel (power-of-two strides past a 16-byte boundary) stages each span
    with 16-byte loads from its first 16-byte boundary and single elements
    around them; the fixed-stride kernel (the other strides) shifts its loads
    to the boundaries.  Spans shorter than the peeled head, spans clipped at n
    and ragged last blocks."""
    L = ew.lib()
    e = ESIZE[dtype]
    ew.set_schedule("tiled")
    try:
        for s in (2, 3, 5, 12, 16, 17, 40, 63, 64):
            for n in (s + 1, s + 2, s + 5, 4097, 70001, (1 << 18) + 3):
                x = inputs.random_bits(n, dtype, 7300 + n + s)
                want = oracle.gather_stride(x, s)
                for in_off in range(16 // e):
                    bi = GuardedBuffer(n, dtype, in_off).fill(x)
                    bo = GuardedBuffer(n, dtype, 1)
                    assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(),
                                              n, s, _stream()) == 0
                    rec = ew.last_launch()
                    assert rec["schedule"] == 4 and rec["vec_bytes"] == 16, (n, s, in_off, rec)
                    torch.cuda.synchronize()
                    assert_bits_equal(bo.host(), want, dtype, False,
                                      "tiled gather n=%d s=%d input offset %d" % (n, s, in_off))
                    assert bi.guards_intact() and bo.guards_intact()
    finally:
        ew.set_schedule("auto")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
def test_gather_auto_crossover(dtype):
    """AUTO's choice around its crossovers: lap order below s = 5 for 4-byte
    elements, the tiled kernels from there (from s = 2 for 2-byte elements)
    to 64, index order from 65; each against the oracle."""
    L = ew.lib()
    ew.set_schedule("auto")
    n = 300_007
    x = inputs.random_bits(n, "f32" if dtype == "i32" else dtype, 7300 + len(dtype))
    for s in (2, 3, 4, 5, 6, 7, 8, 9, 16, 24, 32, 48, 64, 65):
        bi = GuardedBuffer(n, dtype, 0).fill(x)
        bo = GuardedBuffer(n, dtype, 2)
        assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(), n, s, _stream()) == 0
        rec = ew.last_launch()
        assert rec["schedule"] == _gather_auto_schedule(n, s, dtype if dtype != "i32" else "f32"), (s, rec)
        torch.cuda.synchronize()
        assert_bits_equal(bo.host(), oracle.gather_stride(x, s), "f32" if dtype == "i32" else dtype, False,
                          "auto gather %s s=%d" % (dtype, s))
        assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("schedule", ["laps", "tiled"])
@pytest.mark.parametrize("n,s", [(1 << 32, 2), ((1 << 32) - 1, 3), (1 << 32, 64), ((1 << 32) - 7, 5)])
def test_gather_lap_order_at_2p32_int32(n, s, schedule):
    """The lap-ordered and tiled gathers' 32-bit index arithmetic at n <= 2^32:
    the input holds its own index (int32, i.e. modulo 2^32), so every output
    names the source it was read from.  All n outputs are compared with
    (s*i) mod n computed in int64 by torch, chunk by chunk, and 2,000
    positions (both ends, every lap boundary, random) with the oracle's
    128-bit index map."""
    chunk = 1 << 28
    tin = torch.empty(n, dtype=torch.int32, device="cuda")
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        v = torch.arange(lo, hi, dtype=torch.int64, device="cuda")
        tin[lo:hi] = ((v + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
        del v
    tout = torch.empty_like(tin)
    ew.set_schedule(schedule)
    assert ew.lib().ew_gather_stride(3, tin.data_ptr(), tout.data_ptr(), n, s, _stream()) == 0
    rec = ew.last_launch()
    assert rec["schedule"] == (3 if schedule == "laps" else 4), rec
    torch.cuda.synchronize()
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        want = torch.arange(lo, hi, dtype=torch.int64, device="cuda") * s % n
        got = tout[lo:hi].to(torch.int64) % (1 << 32)
        assert torch.equal(got, want), "chunk at %d" % lo
        del want, got
    g = inputs.rng(8300 + s)
    bounds = [-(-lap * n // s) for lap in range(s + 1)]
    idx = sorted({int(i) for b in bounds for i in (b - 1, b, b + 1) if 0 <= i < n}
                 | set(range(0, 200)) | set(range(n - 200, n))
                 | {int(i) for i in g.integers(0, n, size=1500, dtype=np.int64)})
    got = tout[torch.tensor(idx, dtype=torch.int64, device="cuda")].cpu().numpy().view(np.uint32)
    want = np.array([oracle.gather_index(i, s, n) for i in idx], dtype=np.int64)
    assert np.array_equal(got.astype(np.int64), want)
    del tin, tout
    torch.cuda.empty_cache()


@pytest.mark.parametrize("schedule,s", [("laps", 2), ("laps", 5), ("tiled", 3), ("tiled", 16), ("tiled", 64)])
def test_gather_at_2p32_16bit_low_index_bits(schedule, s):
    """The 2-byte lap-ordered and tiled gathers at n = 2^32: element j holds the
    low 16 bits of j, so every output must equal the low 16 bits of
    (s*i) mod n; all 2^32 outputs are compared chunk by chunk (int64 on the
    device), and lap boundaries and random positions against the oracle's
    128-bit index map."""
    n = 1 << 32
    chunk = 1 << 28
    tin = torch.empty(n, dtype=torch.int16, device="cuda")
    for lo in range(0, n, chunk):
        v = torch.arange(lo, lo + chunk, dtype=torch.int64, device="cuda")
        tin[lo:lo + chunk] = ((v & 0xFFFF) - ((v & 0x8000) << 1)).to(torch.int16)
        del v
    tout = torch.empty_like(tin)
    ew.set_schedule(schedule)
    assert ew.lib().ew_gather_stride(1, tin.data_ptr(), tout.data_ptr(), n, s, _stream()) == 0
    assert ew.last_launch()["schedule"] == (3 if schedule == "laps" else 4)
    torch.cuda.synchronize()
    for lo in range(0, n, chunk):
        want = (torch.arange(lo, lo + chunk, dtype=torch.int64, device="cuda") * s % n) & 0xFFFF
        got = tout[lo:lo + chunk].to(torch.int64) & 0xFFFF
        assert torch.equal(got, want), "chunk at %d" % lo
        del want, got
    g = inputs.rng(8400 + s)
    bounds = [-(-lap * n // s) for lap in range(s + 1)]
    idx = sorted({int(i) for b in bounds for i in (b - 1, b, b + 1) if 0 <= i < n}
                 | set(range(0, 100)) | set(range(n - 100, n))
                 | {int(i) for i in g.integers(0, n, size=1000, dtype=np.int64)})
    got = tout[torch.tensor(idx, dtype=torch.int64, device="cuda")].cpu().numpy().view(np.uint16)
    want = np.array([oracle.gather_index(i, s, n) & 0xFFFF for i in idx], dtype=np.uint16)
    assert np.array_equal(got, want)
    del tin, tout
    torch.cuda.empty_cache()


def _random_i32(n, seed):
    g = inputs.rng(seed)
    x = g.integers(-2 ** 31, 2 ** 31, size=n, dtype=np.int64).astype(np.int32)
    if n:
        x[: min(n, 6)] = np.array([0, 1, -1, 2 ** 31 - 1, -2 ** 31, 2 ** 30], dtype=np.int32)[: min(n, 6)]
    return x


@pytest.mark.parametrize("schedule", ["oneshot", "persistent"])
@pytest.mark.parametrize("path", PATHS)
def test_select_even_odd_i32(path, schedule):
    """y = x even ? 2x : x + 1 on int32 at every width, offset, ragged size and
    schedule, out of place and in place."""
    L = ew.lib()
    ew.set_path(path)
    ew.set_schedule(schedule)
    for n in (1, 5, 8, 9, 33, 1000, 4099, 70001, 600_001):
        for off in (0, 1, 3):
            x = _random_i32(n, 9300 + n + off)
            want = oracle.select_even_odd(x)
            bx = GuardedBuffer(n, "i32", off).fill(x)
            by = GuardedBuffer(n, "i32", off)
            assert L.ew_select_even_odd(3, bx.view.data_ptr(), by.view.data_ptr(), n, _stream()) == 0
            torch.cuda.synchronize()
            assert np.array_equal(by.host(), want), (path, schedule, n, off)
            assert L.ew_select_even_odd(3, bx.view.data_ptr(), bx.view.data_ptr(), n, _stream()) == 0
            torch.cuda.synchronize()
            assert np.array_equal(bx.host(), want), ("in place", path, schedule, n, off)
            assert bx.guards_intact() and by.guards_intact()


def test_select_even_odd_i32_2p28_and_int32_copy_gather():
    n = 1 << 28
    x = _random_i32(n, 9400)
    bx = GuardedBuffer(n, "i32").fill(x)
    by = GuardedBuffer(n, "i32")
    L = ew.lib()
    assert L.ew_select_even_odd(3, bx.view.data_ptr(), by.view.data_ptr(), n, _stream()) == 0
    torch.cuda.synchronize()
    assert np.array_equal(by.host(), oracle.select_even_odd(x))
    m = 1 << 22
    assert L.ew_copy(3, bx.view.data_ptr(), by.view.data_ptr(), m, _stream()) == 0
    torch.cuda.synchronize()
    assert np.array_equal(by.host()[:m], x[:m])
    assert L.ew_gather_stride(3, bx.view.data_ptr(), by.view.data_ptr(), m, 2, _stream()) == 0
    torch.cuda.synchronize()
    assert np.array_equal(by.host()[:m], oracle.gather_stride(x[:m], 2))
    assert by.guards_intact()


def test_binding_select_even_odd():
    x = torch.from_numpy(_random_i32(10_001, 9500)).cuda()
    y = ew.ew_select_even_odd(x)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.select_even_odd(x.cpu().numpy()))
    with pytest.raises(ew.EwError):
        ew.ew_select_even_odd(x.float())


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_gather_span_variant(dtype):
    """ew_set_path(v256): strides 2 and 4 load contiguous source spans and
    select every stride-th word; other strides keep one load per output.
    Sizes with and without wrap-around, input and output offsets that keep or
    break the 32-byte span alignment."""
    L = ew.lib()
    code = DT_CODE.get(dtype, 3)
    ew.set_path("v256")
    for n in (3, 5, 9, 17, 64, 1000, 4096, 4099, 65536, 300_001, 1 << 22):
        x = inputs.random_bits(n, "f32", 9600 + n)
        for s in (2, 4, 3, n + 2):
            for in_off, out_off in ((0, 0), (1, 0), (0, 3), (2, 5)):
                bi = GuardedBuffer(n, dtype, in_off).fill(x)
                bo = GuardedBuffer(n, dtype, out_off)
                assert L.ew_gather_stride(code, bi.view.data_ptr(), bo.view.data_ptr(), n, s, _stream()) == 0
                rec = ew.last_launch()
                span = (s % n) in (2, 4)
                assert rec["path"] == (3 if span else 1), (n, s, rec)
                torch.cuda.synchronize()
                assert_bits_equal(bo.host(), oracle.gather_stride(x, s), "f32", False,
                                  "span gather n=%d s=%d offs=%d,%d" % (n, s, in_off, out_off))
                assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
def test_gather_tiled_pow2(dtype):
    """The tiled gather specialised for strides 2, 4, 8, 16, 32 and 64 (and
    strides congruent to them mod n), on a 16-byte aligned input (strides 2
    and 4 under EW_SCHED_TILED, the others under AUTO): one ragged block,
    exactly one and several full 16 KiB spans, spans plus a ragged block, n
    divisible by the stride (every lap on one residue row) and not (laps of
    unequal length on distinct rows), output offsets that start laps on odd
    and even elements (16-bit runs stored as words or as halves).  A 2-byte
    input offset takes the general tiled kernel."""
    L = ew.lib()
    code = DT_CODE[dtype]
    e = ESIZE[dtype]
    span = 16384 // e  # input elements a block stages (16 KiB)
    bits = "f32" if dtype == "i32" else dtype
    for s in (2, 4, 8, 16, 32, 64):
        ew.set_schedule("tiled" if s < 8 else "auto")
        sizes = (s + 1, 1000, span - 1, span, span + 1, 2 * span, 3 * span + 5, (1 << 20) + 3, 1 << 20)
        for n in sizes:
            x = inputs.random_bits(n, bits, 9900 + n + s)
            for stride in ((s, n + s) if n < 2000 else (s,)):
                for in_off, out_off in ((0, 0), (0, 1), (0, 3), (4 // e if e == 2 else 1, 2)):
                    bi = GuardedBuffer(n, dtype, in_off).fill(x)
                    bo = GuardedBuffer(n, dtype, out_off)
                    assert L.ew_gather_stride(code, bi.view.data_ptr(), bo.view.data_ptr(), n, stride,
                                              _stream()) == 0
                    rec = ew.last_launch()
                    aligned = (in_off * e) % 16 == 0
                    assert rec["schedule"] == 4, (n, s, rec)
                    assert rec["path"] == 2 and rec["vec_bytes"] == 16, rec  # general kernel too: 16-byte staging
                    if aligned:
                        assert rec["grid"] == -(-(-(-n // s)) // (span // s)), (n, s, rec)
                    torch.cuda.synchronize()
                    assert_bits_equal(bo.host(), oracle.gather_stride(x, stride), bits, False,
                                      "pow2 tiled gather %s n=%d s=%d offs=%d,%d"
                                      % (dtype, n, stride, in_off, out_off))
                    assert bi.guards_intact() and bo.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("s", [16, 64])
def test_gather_pow2_full_size_2p26(dtype, s):
    """The bench's tiled gathers at n = 2^26, every output against the oracle."""
    n = 1 << 26
    x = inputs.as_dtype(inputs.uniform(n, inputs.seed_for("copy_f32", 3), 0.0, 1.0), dtype)
    bi, bo = GuardedBuffer(n, dtype).fill(x), GuardedBuffer(n, dtype)
    assert ew.lib().ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(), n, s,
                                     _stream()) == 0
    rec = ew.last_launch()
    assert rec["schedule"] == 4 and rec["path"] == 2, rec
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False, "gather %d 2^26 %s" % (s, dtype))
    assert bo.guards_intact() and bi.guards_intact()


@pytest.mark.parametrize("dtype,s,in_off", [("f32", 63, 0), ("bf16", 33, 0), ("bf16", 6, 0), ("f32", 12, 0),
                                           ("f32", 40, 1), ("bf16", 17, 3), ("bf16", 6, 7), ("f32", 16, 1),
                                           ("bf16", 64, 5), ("bf16", 4, 3)])
def test_gather_fixed_and_general_full_size_2p26(dtype, s, in_off):
    """The fixed-stride kernel at n = 2^26 (s = 63 and 33 with a partial last
    warp, s = 6 and 12 with the larger register allowance, s = 40, 17 and 6 on
    inputs 1, 3 and 7 elements past 16 bytes) and the general kernel (power-of-
    two strides on inputs past 16 bytes, but 2-byte elements at s = 4, which
    take the fixed-stride kernel's shifted instance): every output against the
    oracle, with the block size the launch record reports."""
    n = 1 << 26
    e = ESIZE[dtype]
    x = inputs.as_dtype(inputs.uniform(n, inputs.seed_for("copy_f32", 5), 0.0, 1.0), dtype)
    bi, bo = GuardedBuffer(n, dtype, in_off).fill(x), GuardedBuffer(n, dtype)
    assert ew.lib().ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(), n, s,
                                     _stream()) == 0
    rec = ew.last_launch()
    assert rec["schedule"] == 4 and rec["path"] == 2, rec
    # aligned powers of two: the power-of-two kernel; past 16 bytes the general
    # kernel (both 256 threads), but for 2-byte elements at s = 2, 4, 8; every
    # other case the fixed-stride one
    pow2, aligned = s & (s - 1) == 0, (in_off * e) % 16 == 0
    shifted_pow2 = pow2 and not aligned and e == 2 and s <= 8
    assert rec["block"] == (256 if pow2 and not shifted_pow2 else fixed_block(s, e)), rec
    torch.cuda.synchronize()
    assert_bits_equal(bo.host(), oracle.gather_stride(x, s), dtype, False,
                      "gather %d 2^26 %s offset %d" % (s, dtype, in_off))
    assert bo.guards_intact() and bi.guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "i32"])
def test_gather_random_cases(dtype):
    """Seeded random gathers across every schedule: sizes from 1 to 2^20 + 999
    (ragged tiles and laps), strides from 1 to 200 and beyond n, input and
    output offsets from 0 to 9 elements; each output against the oracle and
    the guard zones intact."""
    L = ew.lib()
    g = inputs.rng(0x6A7E + DT_CODE[dtype])
    bits = "f32" if dtype == "i32" else dtype
    for case in range(60):
        n = int(g.choice([g.integers(1, 5000), g.integers(5000, 300_000), g.integers(300_000, (1 << 20) + 1000)]))
        s = int(g.choice([g.integers(1, 9), g.integers(9, 65), g.integers(65, 200), n + int(g.integers(0, 70))]))
        sched = str(g.choice(["auto", "auto", "laps", "tiled", "oneshot", "persistent"]))
        in_off, out_off = int(g.integers(0, 10)), int(g.integers(0, 10))
        ew.set_schedule(sched)
        x = inputs.random_bits(n, bits, 12000 + case)
        bi = GuardedBuffer(n, dtype, in_off).fill(x)
        bo = GuardedBuffer(n, dtype, out_off)
        assert L.ew_gather_stride(DT_CODE[dtype], bi.view.data_ptr(), bo.view.data_ptr(), n, s, _stream()) == 0
        torch.cuda.synchronize()
        assert_bits_equal(bo.host(), oracle.gather_stride(x, s), bits, False,
                          "random gather %s n=%d s=%d %s offs=%d,%d" % (dtype, n, s, sched, in_off, out_off))
        assert bi.guards_intact() and bo.guards_intact()
    ew.set_schedule("auto")


FIXED_STRIDES = tuple(s for s in range(3, 64) if s & (s - 1))  # every stride up to 63 but the powers of two


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
def test_gather_tiled_fixed_strides(dtype):
    """The tiled gather specialised for fixed strides that are not powers of
    two (every stride from 3 to 63 but 4, 8, 16, 32, and strides congruent to
    them mod n) on a
    16-byte aligned input, with the block size chosen per stride: one ragged
    block, one and several full spans, spans plus a ragged block, n divisible
    by the stride and not, output offsets that start laps on odd and even
    elements.  An input offset of 2 or 4 bytes runs the same kernel with its
    loads shifted to the 16-byte boundaries."""
    L = ew.lib()
    code = DT_CODE[dtype]
    e = ESIZE[dtype]
    bits = "f32" if dtype == "i32" else dtype
    ew.set_schedule("tiled")
    for s in FIXED_STRIDES:
        for n in (s + 1, 997, 4096 * 4 // e - 1, 16384 // e + 5, 3 * 16384 // e + 11, (1 << 20) + 3, 1 << 20):
            x = inputs.random_bits(n, bits, 15000 + n + s)
            for stride in ((s, n + s) if n < 2000 else (s,)):
                for in_off, out_off in ((0, 0), (0, 1), (0, 3), (4 // e if e == 2 else 1, 2)):
                    bi = GuardedBuffer(n, dtype, in_off).fill(x)
                    bo = GuardedBuffer(n, dtype, out_off)
                    assert L.ew_gather_stride(code, bi.view.data_ptr(), bo.view.data_ptr(), n, stride,
                                              _stream()) == 0
                    rec = ew.last_launch()
                    aligned = (in_off * e) % 16 == 0
                    assert rec["schedule"] == 4, (n, s, rec)
                    assert rec["path"] == 2 and rec["vec_bytes"] == 16, rec  # general kernel too: 16-byte staging
                    assert rec["block"] == fixed_block(s, e), rec  # any offset: shifted loads
                    torch.cuda.synchronize()
                    assert_bits_equal(bo.host(), oracle.gather_stride(x, stride), bits, False,
                                      "fixed tiled gather %s n=%d s=%d offs=%d,%d"
                                      % (dtype, n, stride, in_off, out_off))
                    assert bi.guards_intact() and bo.guards_intact()
    ew.set_schedule("auto")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gather_plan_query_matches_the_launch(dtype):
    """ew_gather_plan_query reports the launch record a real ew_gather_stride
    call leaves, for each schedule, aligned and offset inputs and strides
    taking each kernel (the grid-stride kernel's grid aside: the query leaves
    it to the device)."""
    L = ew.lib()
    code = DT_CODE[dtype]
    n = 300_007
    x = inputs.random_bits(n, dtype, 7800)
    try:
        for sched in ("auto", "tiled", "laps", "oneshot", "persistent"):
            ew.set_schedule(sched)
            for s in (2, 3, 4, 8, 12, 16, 33, 64, 65):
                for in_off in (0, 1, 3):
                    bi = GuardedBuffer(n, dtype, in_off).fill(x)
                    bo = GuardedBuffer(n, dtype, 0)
                    want = ew.gather_plan_query(code, bi.view.data_ptr(), bo.view.data_ptr(), n, s)
                    assert L.ew_gather_stride(code, bi.view.data_ptr(), bo.view.data_ptr(), n, s,
                                              _stream()) == 0
                    got = ew.last_launch()
                    if got["schedule"] == 2:
                        assert want["grid"] == 0 and got["grid"] > 0
                        want["grid"] = got["grid"]
                    assert got == want, (sched, s, in_off, got, want)
            torch.cuda.synchronize()
    finally:
        ew.set_schedule("auto")
