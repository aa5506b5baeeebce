"""Streams, threads and CUDA graphs around the C ABI.

The library launches on the caller's stream and never synchronises, so it
must work from several host threads at once, on non-default streams, and
inside a captured CUDA graph (no synchronising or allocating call on the
launch path).
"""
import threading

import numpy as np
import pytest
import torch

import memory_bound_elementwise_gb300 as ew
import oracle
from memory_bound_elementwise_gb300 import inputs
from tests.gpu_util import assert_bits_equal

pytestmark = pytest.mark.gpu


def _f32(n, seed):
    return inputs.uniform(n, seed)


def test_many_threads_many_streams():
    n = (1 << 20) + 7
    nthreads = 8
    host = [(_f32(n, 100 + t), _f32(n, 200 + t)) for t in range(nthreads)]
    want = [oracle.add("f32", a, b) for a, b in host]
    results = [None] * nthreads
    errors = []

    def worker(t):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                a = torch.from_numpy(host[t][0]).cuda(non_blocking=False)
                b = torch.from_numpy(host[t][1]).cuda(non_blocking=False)
                c = torch.empty_like(a)
                for _ in range(20):  # repeated launches interleave with the other threads
                    ew.ew_add(a, b, c, stream=s)
                    rec = ew.last_launch()  # per-thread record
                    assert rec["launches"] == 1 and rec["nvec"] == n // 8
                s.synchronize()
                results[t] = c.cpu().numpy()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    ths = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
    assert not errors, errors
    for t in range(nthreads):
        assert_bits_equal(results[t], want[t], "f32", True, "thread %d" % t)


def test_stream_ordering_between_calls():
    """relu(a + b) as two calls on one non-default stream, then read on another
    stream after an event: the second call sees the first one's output."""
    n = 3_000_001
    a, b = _f32(n, 300), _f32(n, 301)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    torch.cuda.synchronize()
    c = torch.empty_like(ta)
    ew.ew_add(ta, tb, c, stream=s1)
    ew.ew_relu(c, c, stream=s1)
    ev = torch.cuda.Event()
    ev.record(s1)
    s2.wait_event(ev)
    with torch.cuda.stream(s2):
        out = c.clone()
    s2.synchronize()
    want = oracle.relu("f32", oracle.add("f32", a, b))
    assert_bits_equal(out.cpu().numpy(), want, "f32", False, "add then relu")


@pytest.mark.parametrize("path", ["auto", "tma"])
def test_cuda_graph_capture_and_replay(path):
    n = (1 << 22) + 5
    ew.set_path(path)
    try:
        a = torch.empty(n, device="cuda")
        b = torch.empty(n, device="cuda")
        c = torch.empty(n, device="cuda")
        y = torch.empty(n, device="cuda")
        s = torch.cuda.Stream()
        # one eager call first (fills the per-device caches)
        ew.ew_add(a.zero_(), b.zero_(), c, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ew.ew_add(a, b, c, stream=s)
            ew.ew_saxpy(2.5, c, y, stream=s)
            ew.ew_relu(y, y, stream=s)
        for rep in range(3):
            ha, hb, hy = _f32(n, 400 + rep), _f32(n, 500 + rep), _f32(n, 600 + rep)
            a.copy_(torch.from_numpy(ha))
            b.copy_(torch.from_numpy(hb))
            y.copy_(torch.from_numpy(hy))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            want_c = oracle.add("f32", ha, hb)
            want_y = oracle.relu("f32", oracle.saxpy("f32", 2.5, want_c, hy))
            assert_bits_equal(c.cpu().numpy(), want_c, "f32", True, "graph add rep %d" % rep)
            assert_bits_equal(y.cpu().numpy(), want_y, "f32", False, "graph chain rep %d" % rep)
    finally:
        ew.set_path("auto")
    assert ew.device_error() == (0, 0)


def test_graph_capture_of_gathers():
    """Every gather kernel AUTO picks, captured into one CUDA graph: lap order
    (fp32, s = 2), the general tiled kernel (fp32, s = 12), the specialised
    tiled kernels (fp32, s = 16; bf16, s = 2, whose store packs 16-bit pairs)
    and index order (s = 65); replayed on fresh inputs against the oracle."""
    n = (1 << 21) + 9
    x = torch.empty(n, device="cuda")
    xh = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    outs = {s: torch.empty(n, device="cuda") for s in (2, 12, 16, 65)}
    out_h = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for s, o in outs.items():
            ew.ew_gather_stride(x, o, s, stream=st)
        ew.ew_gather_stride(xh, out_h, 2, stream=st)
    for rep in range(2):
        hx = _f32(n, 700 + rep)
        hh = inputs.as_dtype(_f32(n, 800 + rep), "bf16")
        x.copy_(torch.from_numpy(hx))
        xh.copy_(torch.from_numpy(hh.view("int16")).view(torch.bfloat16))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for s, o in outs.items():
            assert_bits_equal(o.cpu().numpy(), oracle.gather_stride(hx, s), "f32", False,
                              "graph gather s=%d rep %d" % (s, rep))
        got_h = out_h.view(torch.int16).cpu().numpy().view("uint16")
        assert_bits_equal(got_h, oracle.gather_stride(hh, 2), "bf16", False, "graph bf16 gather rep %d" % rep)


def test_graph_capture_of_mixed_parity_bf16_add():
    """A 16-bit add with pointers of different parity, captured into a graph:
    inside the capture AUTO keeps the vector kernel (no pointer queries while
    capturing); eager calls on the same buffers take the realigning bulk copy.
    Both give the oracle's bits."""
    n = (1 << 22) + 3
    x = inputs.as_dtype(inputs.normal(n + 8, 720), "bf16")
    y = inputs.as_dtype(inputs.normal(n + 8, 721), "bf16")
    tx = torch.from_numpy(x.view(np.int16)).cuda()
    ty = torch.from_numpy(y.view(np.int16)).cuda()
    tz = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    L = ew.lib()
    want = oracle.add("bf16", x[1:1 + n], y[:n])
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert L.ew_add(2, tx.data_ptr() + 2, ty.data_ptr(), tz.data_ptr() + 6, n, s.cuda_stream) == 0
        rec = ew.last_launch()
    assert rec["path"] != 4 and rec["vec_bytes"] == 2, rec
    g.replay()
    torch.cuda.synchronize()
    assert_bits_equal(tz.cpu().numpy().view(np.uint16)[3:3 + n], want, "bf16", True, "captured mixed parity")
    tz.zero_()
    assert L.ew_add(2, tx.data_ptr() + 2, ty.data_ptr(), tz.data_ptr() + 6, n,
                    torch.cuda.current_stream().cuda_stream) == 0
    assert ew.last_launch()["path"] == 4
    torch.cuda.synchronize()
    assert_bits_equal(tz.cpu().numpy().view(np.uint16)[3:3 + n], want, "bf16", True, "eager mixed parity")


def test_bf16_tensor_views_with_offsets():
    """Binding on sliced views: data_ptr carries the element offset."""
    n = 1 << 20
    base_a = inputs.as_dtype(inputs.normal(n + 3, 700), "bf16")
    base_b = inputs.as_dtype(inputs.normal(n + 3, 701), "bf16")
    ta = torch.from_numpy(base_a.view(np.int16)).cuda().view(torch.bfloat16)
    tb = torch.from_numpy(base_b.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty(n + 3, dtype=torch.bfloat16, device="cuda")
    ew.ew_add(ta[3:], tb[1:n + 1], out[2:n + 2])
    rec = ew.last_launch()
    torch.cuda.synchronize()
    got = out[2:n + 2].view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.add("bf16", base_a[3:], base_b[1:n + 1])
    assert_bits_equal(got, want, "bf16", True, "bf16 views")
    # offsets 6, 2 and 4 bytes agree only modulo 2: one element per access
    assert rec["vec_bytes"] == 2


@pytest.mark.parametrize("programmatic", [True, False])
@pytest.mark.parametrize("path", ["auto", "tma"])
def test_dependent_chain_of_calls(programmatic, path):
    """Sixty rounds of SAXPY -> ReLU in place -> add -> copy -> gather on one
    stream, each call reading what the previous one wrote, with programmatic
    dependent launch on and off: the result must equal the oracle applied
    round by round."""
    n = (1 << 18) + 3
    x = inputs.normal(n, 9700)
    y = inputs.normal(n, 9701)
    ew.set_programmatic_launch(programmatic)
    ew.set_path(path)
    try:
        tx, ty = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
        tz, tw = torch.empty_like(tx), torch.empty_like(tx)
        torch.cuda.synchronize()
        hx, hy = x.copy(), y.copy()
        for _ in range(60):
            ew.ew_saxpy(0.75, tx, ty)
            ew.ew_relu(ty, ty)
            ew.ew_add(ty, tx, tz)
            ew.ew_copy(tz, ty)
            ew.ew_gather_stride(ty, tw, 3)
            ew.ew_add(tw, tx, ty)
            hy = oracle.relu("f32", oracle.saxpy("f32", 0.75, hx, hy))
            hz = oracle.add("f32", hy, hx)
            hw = oracle.gather_stride(hz, 3)
            hy = oracle.add("f32", hw, hx)
        torch.cuda.synchronize()
        assert_bits_equal(ty.cpu().numpy(), hy, "f32", True, "dependent chain")
    finally:
        ew.set_programmatic_launch(True)
        ew.set_path("auto")
    assert ew.device_error() == (0, 0)
