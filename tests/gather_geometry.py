"""The tiled gathers' block geometry, stated independently of the library:
threads per block, loads per thread and lap positions per block P, for the
fixed-stride kernel (s not a power of two, and 16-bit s = 2, 4, 8 on an input
past a 16-byte boundary), the power-of-two kernel and the general kernel.
Shared by the host-side plan tests and the GPU parity tests."""
import math


def fixed_geometry(s, e):
    """(threads T, 16-byte loads per thread) of the fixed-stride kernel.  T is
    a multiple of the row period s / gcd(s, V) (V = 16 / e elements per load),
    so that a thread's rows stay fixed across its loads.  Whole warps: the
    smallest multiple of lcm(32, period) from 192 (384 from s = 32), if at most
    512; else the multiple of the period up to 512 whose span (loads x 16 x T)
    comes nearest its target, whole warps breaking ties.  Loads: from the
    target's worth (16 KiB; 20 KiB for 352 threads or more; 24 KiB for 480; 32
    KiB from s = 32) up, the first count that gives each warp's share of a lap
    run a whole number of warp-wide 4-byte words."""
    v = 16 // e
    period = s // math.gcd(s, v)
    least = 384 if s >= 32 else 192
    align = 64 if e == 2 else 32

    def target(t):
        return 32768 if s >= 32 else 24576 if t >= 480 else 20480 if t >= 352 else 16384

    def loads(t):
        wpl = 1 if s >= t // 32 else (t // 32) // s
        for n_loads in range(max(target(t) // (16 * t), 1), 65):
            if (n_loads * v * t // s) % (align * wpl) == 0:
                return n_loads
        return None

    lcm = math.lcm(32, period)
    whole = -(-least // lcm) * lcm
    if whole <= 512:
        return whole, loads(whole)

    def deviation(t):
        n_loads = loads(t)
        return 1 << 30 if n_loads is None else abs(n_loads * 16 * t - target(t))
    best = None
    for t in range(-(-least // period) * period, 513, period):
        if best is None or deviation(t) < deviation(best) or (
                deviation(t) == deviation(best) and t % 32 == 0 and best % 32 != 0):
            best = t
    return best, loads(best)


def fixed_block(s, e):
    return fixed_geometry(s, e)[0]


def fixed_positions(s, e):
    """Lap positions per block of the fixed-stride kernel: its span over s."""
    t, n_loads = fixed_geometry(s, e)
    return n_loads * (16 // e) * t // s


def pow2_positions(s, e):
    """The power-of-two kernel stages 16 KiB per block."""
    return 16384 // e // s


def general_positions(s, e):
    """The general kernel: the largest power of two P with s*P*e <= 20 KiB,
    raised until a lap run (P*e bytes) is at least 512 bytes."""
    log2p = 0
    while (2 << log2p) * s * e <= 20480:
        log2p += 1
    while (1 << log2p) * e < 512:
        log2p += 1
    return 1 << log2p
