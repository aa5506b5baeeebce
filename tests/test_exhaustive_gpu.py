"""Every pair of 16-bit operands through the GPU's packed add, its SAXPY
(alpha = 2.5, the pages' coefficient) and the fused SAXPY + ReLU: 2^32 pairs
per format and operator, in 16 launches of 2^28, compared with the oracle bit
for bit (for the fused operator: the oracle's saxpy, then its relu); NaN
results compare as "both NaN".  About 35 s per operator on a GB300 with a
16-core host.

The oracle runs in a pool of worker processes started with "spawn" (never
forked from a process that has touched the GPU).
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import memory_bound_elementwise_gb300 as ew
from tests.gpu_util import is_nan_bits

pytestmark = pytest.mark.gpu

CHUNKS = 16
PER = (1 << 32) // CHUNKS          # pairs per launch
B_PER_CHUNK = PER >> 16           # 4096 distinct B patterns per launch


ALPHA = 2.5


def _oracle_slice(args):
    op, dtype, b_lo, b_hi = args
    import oracle
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bvals = np.arange(b_lo, b_hi, dtype=np.uint32).astype(np.uint16)
    a = np.tile(allp, bvals.size)
    b = np.repeat(bvals, allp.size)
    if op == "add":
        return oracle.add(dtype, a, b)
    if op == "saxpy_relu":
        return oracle.relu(dtype, oracle.saxpy(dtype, ALPHA, a, b))
    return oracle.saxpy(dtype, ALPHA, a, b)  # x = every pattern, y = B


@pytest.mark.parametrize("op", ["add", "saxpy", "saxpy_relu"])
@pytest.mark.parametrize("dtype,code", [("f16", 1), ("bf16", 2)])
def test_all_operand_pairs(op, dtype, code):
    workers = min(16, os.cpu_count() or 4)
    ctx = mp.get_context("spawn")
    allp = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16).cuda()
    a = allp.repeat(B_PER_CHUNK)
    c = torch.empty_like(a)
    L = ew.lib()
    s = torch.cuda.current_stream().cuda_stream
    with ctx.Pool(workers) as pool:
        for chunk in range(CHUNKS):
            b_lo = chunk * B_PER_CHUNK
            bvals = torch.arange(b_lo, b_lo + B_PER_CHUNK, dtype=torch.int32).to(torch.int16).cuda()
            b = bvals.repeat_interleave(1 << 16)
            if op == "add":
                assert L.ew_add(code, a.data_ptr(), b.data_ptr(), c.data_ptr(), PER, s) == 0
            elif op == "saxpy":
                c.copy_(b)
                assert L.ew_saxpy(code, ALPHA, a.data_ptr(), c.data_ptr(), PER, s) == 0
            else:
                c.copy_(b)
                assert L.ew_saxpy_relu(code, ALPHA, a.data_ptr(), c.data_ptr(), PER, s) == 0
            step = B_PER_CHUNK // workers
            parts = pool.map(_oracle_slice, [(op, dtype, b_lo + k * step, b_lo + (k + 1) * step)
                                             for k in range(workers)])
            want = np.concatenate(parts)
            torch.cuda.synchronize()
            got = c.cpu().numpy().view(np.uint16)
            gn, wn = is_nan_bits(got, dtype), is_nan_bits(want, dtype)
            bad = np.nonzero((got != want) & ~(gn & wn))[0]
            assert bad.size == 0, "%s %s chunk %d: %d mismatches, first pair index %d" % (
                op, dtype, chunk, bad.size, int(bad[0]))
