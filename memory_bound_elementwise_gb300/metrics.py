"""Algorithmic byte counts and bandwidth arithmetic for the benchmark.

Bytes are the ones the operation must move at least once, counted per element:

* add     C = A + B        read A, read B, write C   -> 3 element transfers
  ("逐元素操作算子" §一.2: 12 bytes per binary32 add, 1 FLOP / 12 B;
  "HyperAI elementwise add on RTX 5090", benchmark script: 3 * numel * elsize)
* saxpy   y = a*x + y      read x, read y, write y   -> 3
  ("Puzzle 31", single-pass analysis: 2 reads + 1 write of 32M binary32 = 384 MB)
* relu    y = max(x, 0)    read x, write y           -> 2
  (CUDA-MODE lecture notes §5.2 example 1, case A: 4 B read + 4 B written)
* copy    out = in         read in, write out        -> 2
* add_relu C = max(A + B, 0), fused: 3, against 3 + 2 for the two passes
  (CUDA-MODE lecture notes §5.3, kernel fusion)
* saxpy_relu y = max(a*x + y, 0), fused: 3, against 3 + 2 for the two passes
* select  y = x even ? 2x : x + 1 on int32 -> 2 (CUDA-MODE lecture notes §6)
* gather  out[i] = in[(s*i) mod n]: one element read and one written per
  output -> 2 (logical bytes; the sectors actually fetched are larger and are
  reported separately from the profiler).

GB/s is decimal (10^9 bytes per second), as in the pages' benchmark script.
"""

ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}

TRANSFERS_PER_ELEMENT = {
    "add": 3,
    "add_relu": 3,
    "saxpy_relu": 3,
    "saxpy": 3,
    "relu": 2,
    "copy": 2,
    "gather": 2,
    "select": 2,
}


def algorithmic_bytes(op: str, dtype: str, n: int) -> int:
    return TRANSFERS_PER_ELEMENT[op] * ELEM_SIZE[dtype] * int(n)


def gbps(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / 1e9


def arithmetic_intensity(op: str, dtype: str) -> float:
    """FLOP (or compare) per algorithmic byte for one element."""
    flops = {"add": 1, "add_relu": 2, "saxpy": 2, "relu": 1, "copy": 0, "gather": 0, "select": 2}[op]
    return flops / (TRANSFERS_PER_ELEMENT[op] * ELEM_SIZE[dtype])
