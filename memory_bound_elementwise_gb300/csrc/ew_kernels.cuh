// ew_kernels.cuh -- the streaming (load, operate, store) kernel and the
// strided-gather kernels, as templates instantiated per operator and width by
// ew_kernels_{f32,f16,bf16}.cu.
//
// Streaming kernel ("逐元素操作算子" §二: template kernel, grid-stride loop,
// float4 body with scalar tail; "HyperAI elementwise add", Versions 5-6:
// several wide loads in flight per thread):
//   * the body is cut into chunks of kBlock*U vectors; block b takes chunks
//     b, b + gridDim.x, ... (one chunk per block when the grid covers them all);
//   * each thread issues U independent VB-byte loads per input before any
//     arithmetic, then U VB-byte stores, lanes of a warp on consecutive vectors;
//   * the few elements before the first VB-aligned address (head) and after
//     the last whole vector (tail) are done one by one by block 0, in the same
//     launch.
// With one chunk per block (the default "one-shot" schedule) the hardware
// block scheduler hands chunks to whichever SM frees a slot first, which
// balances the SMs at the end of the array; a grid of SMs x resident blocks
// (the "persistent" schedule) walks the same chunks with a grid stride.
#pragma once

#include <cstring>
#include <type_traits>

#include "ew_device.cuh"
#include "ew_internal.h"

namespace ew {

template <class Op> __device__ __forceinline__ Op make_op(float) { return Op{}; }
template <> __device__ __forceinline__ OpSaxpyF32 make_op<OpSaxpyF32>(float a) { return OpSaxpyF32{a}; }
template <> __device__ __forceinline__ OpSaxpyF16 make_op<OpSaxpyF16>(float a) { return OpSaxpyF16{a}; }
template <> __device__ __forceinline__ OpSaxpyBF16 make_op<OpSaxpyBF16>(float a) { return OpSaxpyBF16{a}; }
template <> __device__ __forceinline__ OpSaxpyReluF32 make_op<OpSaxpyReluF32>(float a) { return OpSaxpyReluF32{a}; }
template <> __device__ __forceinline__ OpSaxpyReluF16 make_op<OpSaxpyReluF16>(float a) { return OpSaxpyReluF16{a}; }
template <> __device__ __forceinline__ OpSaxpyReluBF16 make_op<OpSaxpyReluBF16>(float a) {
    return OpSaxpyReluBF16{a};
}

template <class Op, int VB, int U>
__global__ void __launch_bounds__(kBlock) stream_kernel(const StreamArgs a) {
    enter_grid();
    const Op op = make_op<Op>(a.alpha);
    constexpr int E = Op::kElem;
    constexpr int64_t kChunk = static_cast<int64_t>(kBlock) * U;  // vectors per chunk
    const char *in0 = static_cast<const char *>(a.in0);
    const char *in1 = static_cast<const char *>(a.in1);
    char *out = static_cast<char *>(a.out);

    // scalar head [0, head) and tail [tail0, n): fewer than 32 elements in all
    if (blockIdx.x == 0) {
        const int64_t t = threadIdx.x;
        if (t < a.head) apply_one(op, in0, in1, out, t * E);
        if (t < a.n - a.tail0) apply_one(op, in0, in1, out, (a.tail0 + t) * E);
    }

    const int64_t base = a.head * E;
    const char *b0 = in0 + base;
    const char *b1 = (Op::kIn == 2) ? in1 + base : nullptr;
    char *bo = out + base;
    const int64_t nvec = a.nvec;
    const int64_t nchunks = (nvec + kChunk - 1) / kChunk;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int64_t v0 = c * kChunk + threadIdx.x;
        if ((c + 1) * kChunk <= nvec) {  // whole chunk: no bounds checks
            Vec<VB> x[U], y[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                x[j] = ld<VB>(b0 + (v0 + j * kBlock) * VB);
                if constexpr (Op::kIn == 2) y[j] = ld<VB>(b1 + (v0 + j * kBlock) * VB);
                else y[j] = x[j];
            }
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const Vec<VB> z = apply<Op, VB>(op, x[j], y[j]);
                if constexpr (MaySkipUnchanged<Op>::value) {
                    if (a.skip_unchanged && same_bits<VB>(z, x[j])) continue;
                }
                st<VB>(bo + (v0 + j * kBlock) * VB, z);
            }
        } else {  // last, partial chunk
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int64_t v = v0 + j * kBlock;
                if (v < nvec) {
                    const Vec<VB> x = ld<VB>(b0 + v * VB);
                    Vec<VB> y = x;
                    if constexpr (Op::kIn == 2) y = ld<VB>(b1 + v * VB);
                    const Vec<VB> z = apply<Op, VB>(op, x, y);
                    if constexpr (MaySkipUnchanged<Op>::value) {
                        if (a.skip_unchanged && same_bits<VB>(z, x)) continue;
                    }
                    st<VB>(bo + v * VB, z);
                }
            }
        }
    }
}

template <class Op, int VB, int U>
cudaError_t launch_stream(const StreamArgs &a, int grid, cudaStream_t s) {
    return launch_kernel(&stream_kernel<Op, VB, U>, grid, kBlock, 0, s, a);
}

// Loads in flight per thread per input, by width: 64 bytes each.
template <int VB> struct UnrollFor { static constexpr int value = VB >= 32 ? 2 : VB == 16 ? 4 : 8; };

template <class Op, int VB>
constexpr StreamEntry stream_entry() {
    return StreamEntry{reinterpret_cast<const void *>(&stream_kernel<Op, VB, UnrollFor<VB>::value>),
                       &launch_stream<Op, VB, UnrollFor<VB>::value>, UnrollFor<VB>::value};
}
constexpr StreamEntry kNoEntry{nullptr, nullptr, 0};

// ---------------------------------------------------------------- gather
//
// out[i] = in[(s*i) mod n] ("CUDA-MODE lecture notes" §3.2, non-coalesced copy,
// s = 2 on the page).  One output element per access, as on the page, so a
// warp's load touches every s-th element of a span of 32*s elements while its
// store covers 32 consecutive elements.

__device__ __forceinline__ uint64_t addmod_u64(uint64_t a, uint64_t b, uint64_t n) {
    const uint64_t r = a + b;  // a, b < n <= 2^63
    return r >= n ? r - n : r;
}
__device__ __forceinline__ uint64_t mulmod_u64(uint64_t a, uint64_t b, uint64_t n) {
    // a, b < n <= 2^63: doubling and adding stay below 2^64
    uint64_t r = 0;
    while (b != 0) {
        if (b & 1u) r = addmod_u64(r, a, n);
        a = addmod_u64(a, a, n);
        b >>= 1;
    }
    return r;
}

// One-shot gather for n <= 2^32: thread handles outputs i0 + k*kBlock (k < U)
// of its block's chunk.  (s mod n) * i0 < 2^64 is reduced mod n with the
// precomputed m = floor((2^64 - 1) / n): q = floor(x*m / 2^64) undershoots
// floor(x/n) by at most 2, so r = x - q*n needs at most two subtractions of n.
// Later slots add (s*kBlock) mod n with one conditional subtraction.
template <int E, int U>
__global__ void __launch_bounds__(kBlock) gather_oneshot_kernel(const GatherArgs g) {
    enter_grid();
    const char *in = static_cast<const char *>(g.in);
    char *out = static_cast<char *>(g.out);
    const uint64_t n = g.n;
    const uint64_t i0 = static_cast<uint64_t>(blockIdx.x) * (kBlock * U) + threadIdx.x;
    if (i0 >= n) return;
    const uint64_t x = g.s_mod * i0;
    uint64_t j = x - __umul64hi(x, g.barrett_m) * n;
    j = (j >= n) ? j - n : j;
    j = (j >= n) ? j - n : j;
    Vec<E> v[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
        if (i0 + k * kBlock < n) v[k] = ld<E>(in + j * E);
        j = addmod_u64(j, g.step_mod, n);
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
        if (i0 + k * kBlock < n) st<E>(out + (i0 + k * kBlock) * E, v[k]);
}

// Lap-ordered gather for a small stride (2 <= s <= kMaxLaps, n <= 2^32).  As
// i runs from 0 to n - 1 the source (s*i) mod n sweeps the input s times.
// Lap L holds the outputs i in [ceil(L*n/s), ceil((L+1)*n/s)); there the
// source is s*i - L*n = r_L + s*p, with p the position in the lap and
// r_L = s*ceil(L*n/s) - L*n < s, so no reduction mod n is needed.  Block b
// takes chunk b / s of lap b mod s.  The s blocks that the scheduler starts
// side by side then read the same stretch of the input, and each sector comes
// from DRAM once.  In index order each lap fetches the whole input again once
// it no longer fits in L2.  The work is unchanged: one load per output, from
// the same source.
//
// Index arithmetic is 32-bit: with n = q*s + m (q = lap_q, m = lap_m),
// ceil(L*n/s) = L*q + ceil(L*m/s), where L*m < kMaxLaps^2, and every valid
// position, source and output index is below n <= 2^32.  Divisions by s use
// div_magic = floor(2^32 / s) + 1, which over-estimates by at most one.
__device__ __forceinline__ uint32_t div_by_s(uint32_t a, uint32_t s, uint32_t magic) {
    const uint32_t q = __umulhi(a, magic);  // floor(a / s) or one more
    return q * s > a ? q - 1 : q;
}

template <int E, int U>
__global__ void __launch_bounds__(kBlock) gather_laps_kernel(const GatherArgs g) {
    enter_grid();
    const char *in = static_cast<const char *>(g.in);
    char *out = static_cast<char *>(g.out);
    const uint32_t s = static_cast<uint32_t>(g.s_mod);
    const uint32_t k = div_by_s(blockIdx.x, s, g.div_magic);
    const uint32_t lap = blockIdx.x - k * s;
    const uint32_t a0 = lap * g.lap_m, a1 = a0 + g.lap_m;  // L*m, (L+1)*m
    const uint32_t c0 = div_by_s(a0 + s - 1, s, g.div_magic);  // ceil(L*m/s)
    const uint32_t c1 = div_by_s(a1 + s - 1, s, g.div_magic);
    const uint32_t len = g.lap_q + (c1 - c0);  // outputs in this lap
    const uint32_t p0 = k * (kBlock * U) + threadIdx.x;
    if (p0 >= len) return;
    const uint32_t i0 = lap * g.lap_q + c0 + p0;  // first output of this thread
    const uint32_t j0 = (c0 * s - a0) + s * p0;   // its source
    const uint32_t jstep = s * kBlock;
    Vec<E> v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (p0 + u * kBlock < len) v[u] = ld<E>(in + static_cast<size_t>(j0 + u * jstep) * E);
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (p0 + u * kBlock < len) st<E>(out + static_cast<size_t>(i0 + u * kBlock) * E, v[u]);
}

// Tiled gather for a small stride (2 <= s <= kMaxLaps, n <= 2^32): the
// transpose-like schedule.  Block b owns positions [b*P, (b+1)*P) of every
// lap.  Their sources r_L + s*p fill the input span [s*b*P, s*(b+1)*P),
// clipped at n, which the block reads once, coalesced: 16-byte loads from the
// span's first 16-byte boundary on, single elements before it and after the
// last whole vector.  It writes the span to shared memory transposed:
// element j goes to row j mod s, column j / s.  Row r then holds, in position
// order, the sources of every lap with r_L = r, so each lap's outputs leave as
// one coalesced run.  Rows are padded (the pad searched on the host for the
// bank spread of these staging stores).  Unlike the lap kernel, every input
// element is loaded once per block, whether one lap, several or none use it.
template <int E, int U>
__global__ void __launch_bounds__(kBlock) gather_tiled_kernel(const GatherArgs g) {
    enter_grid();
    using W = typename std::conditional<E == 4, uint32_t, uint16_t>::type;
    constexpr uint32_t kPerVec = 16 / E;
    extern __shared__ __align__(16) unsigned char tile_raw[];
    W *tile = reinterpret_cast<W *>(tile_raw);
    __shared__ uint32_t lap_start[kMaxLaps], lap_len[kMaxLaps], lap_row[kMaxLaps];
    W *out = static_cast<W *>(g.out);
    const uint32_t s = static_cast<uint32_t>(g.s_mod);
    const uint32_t P = g.tile_p, pitch = g.tile_pitch;
    const uint32_t p0 = blockIdx.x * P;
    if (threadIdx.x < s) {  // lap L: first output, length, offset of its source row
        const uint32_t L = threadIdx.x;
        const uint32_t a0 = L * g.lap_m;
        const uint32_t c0 = div_by_s(a0 + s - 1, s, g.div_magic);  // ceil(L*m/s)
        const uint32_t c1 = div_by_s(a0 + g.lap_m + s - 1, s, g.div_magic);
        lap_start[L] = L * g.lap_q + c0;
        lap_len[L] = g.lap_q + (c1 - c0);
        lap_row[L] = (c0 * s - a0) * pitch;
    }
    const uint64_t j0 = static_cast<uint64_t>(s) * p0;  // first source of the span
    const uint32_t span = s * P;
    const uint32_t avail = g.n - j0 < span ? static_cast<uint32_t>(g.n - j0) : span;
    const W *src = static_cast<const W *>(g.in) + j0;
    // Elements before the span's first 16-byte boundary (the input pointer is
    // element-aligned, so this is a whole number of elements).
    const uint32_t to16 = ((16u - (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(src)) & 15u)) & 15u) / E;
    const uint32_t h = to16 < avail ? to16 : avail;
    const uint32_t nv = (avail - h) / kPerVec;
    const uint32_t done = h + nv * kPerVec;  // [h, done) is staged by vector loads
    {
        const uint4 *src4 = reinterpret_cast<const uint4 *>(src + h);
        for (uint32_t base = 0; base < nv; base += U * kBlock) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t vi = base + u * kBlock + threadIdx.x;
                if (vi < nv) v[u] = src4[vi];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t vi = base + u * kBlock + threadIdx.x;
                if (vi >= nv) continue;
                const uint32_t j = h + vi * kPerVec;
                const uint32_t c = div_by_s(j, s, g.div_magic);
                uint32_t r = j - c * s;
                uint32_t at = r * pitch + c;  // tile slot of element j
                W w[kPerVec];
                memcpy(w, &v[u], 16);
#pragma unroll
                for (uint32_t k = 0; k < kPerVec; ++k) {
                    tile[at] = w[k];
                    if (++r == s) {  // next column, row 0
                        r = 0;
                        at = at + 1 - (s - 1) * pitch;
                    } else {
                        at += pitch;
                    }
                }
            }
        }
    }
    // Single elements: the head [0, h) and the ragged end [done, avail), fewer
    // than 2 * kPerVec in all.  (Loading them ahead of the vector loads made
    // this kernel 1-3% slower.)
    const uint32_t rest = h + (avail - done);
    if (threadIdx.x < rest) {
        const uint32_t j = threadIdx.x < h ? threadIdx.x : done + (threadIdx.x - h);
        const uint32_t c = div_by_s(j, s, g.div_magic);
        tile[(j - c * s) * pitch + c] = src[j];
    }
    __syncthreads();
    // Store phase: the block's s lap runs are shared out among its warps (one
    // warp per run, or two or four per run when s is below the warp count);
    // lane l copies positions l, l + 32, ... of its share.  16-bit runs that
    // start on a 4-byte boundary move as 4-byte words (rows start on whole
    // words: the pitch is even for 2-byte elements).
    constexpr uint32_t kWarps = kBlock / 32;
    const uint32_t wpl = s >= kWarps ? 1u : kWarps / s >= 4 ? 4u : kWarps / s >= 2 ? 2u : 1u;
    const uint32_t seg = P / wpl;
    const uint32_t lane = threadIdx.x & 31u;
    for (uint32_t item = threadIdx.x >> 5; item < s * wpl; item += kWarps) {
        const uint32_t L = item / wpl, q0 = (item - L * wpl) * seg;
        const uint32_t len = lap_len[L] > p0 ? min(lap_len[L] - p0, P) : 0u;
        const uint32_t end = len > q0 ? min(len - q0, seg) : 0u;
        const W *row = tile + lap_row[L] + q0;
        W *dst = out + (static_cast<size_t>(lap_start[L]) + p0 + q0);
        if (E == 2 && end == seg && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
            const uint32_t *row_w = reinterpret_cast<const uint32_t *>(row);
            uint32_t *dst_w = reinterpret_cast<uint32_t *>(dst);
#pragma unroll 4
            for (uint32_t w = lane; w < seg / 2; w += 32) dst_w[w] = row_w[w];
        } else {
#pragma unroll 4
            for (uint32_t q = lane; q < end; q += 32) dst[q] = row[q];
        }
    }
}

// Tiled gather for a power-of-two stride S (2 <= S <= 64) known at compile
// time, and an input aligned to 16 bytes.  Same schedule as the tiled kernel
// above: block b owns positions [b*P, (b+1)*P) of every lap and stages the
// input span they draw from.  With S a compile-time power of two every
// division by S is a shift, and a thread's 16-byte loads all land in the
// same rows: thread t's load i holds the span elements j = V*t + V*T*i
// (V elements per load, T threads), i.e. rows (V*t) mod S onwards and column
// (V*t) / S + i*V*T/S, so its shared-memory stores use one base address and
// compile-time offsets.  When S >= V each element of a load goes to its own
// row; the rows are padded (and, from row 32 on, shifted) so that the 32
// lanes of a warp storing element k of their loads hit 32 different banks,
// with the layout found at compile time.  When S < V a load holds V/S
// consecutive columns of every row, which the thread packs and stores as one
// 4- or 8-byte access per row (lanes then write consecutive words).  The
// store phase splits the S lap runs of the block among its warps (a warp per
// lap, or several per lap when S is below the warp count): lane l copies
// positions l, l + 32, ... of its share of a run from one row, 4-byte words
// where the run allows (pairs of 16-bit elements), in a fully unrolled loop.
// The last block, whose span is cut short by n, stages and stores element by
// element with bounds checks.
struct TiledLayout {
    uint32_t pad;  // elements added to every row
    uint32_t x;    // elements added per 32 rows
};

template <int E, int S, int kSpanBytes>
constexpr TiledLayout tiled_pow2_layout() {
    constexpr uint32_t kPerVec = 16 / E, kP = (kSpanBytes / E) / S, kStep = E == 2 ? 2 : 1;
    // S < kPerVec: packed row stores, lanes on consecutive words, no padding needed
    constexpr uint32_t kPadEnd = S < static_cast<int>(kPerVec) ? kStep : 32;
    for (uint32_t pad = 0; pad < kPadEnd; pad += kStep) {
        for (uint32_t x = 0; x < 64; x += kStep) {
            uint32_t banks = 0, words[32] = {};
            bool ok = true;
            for (uint32_t t = 0; t < 32 && ok && S >= static_cast<int>(kPerVec); ++t) {
                const uint32_t j = kPerVec * t, row = j % S, col = j / S;
                const uint32_t word = ((row * (kP + pad) + x * (row >> 5) + col) * E) / 4;
                bool same_word = false;  // two halves of one word: one access
                for (uint32_t q = 0; q < t; ++q) same_word = same_word || words[q] == word;
                words[t] = word;
                if (same_word) continue;
                ok = (banks >> (word % 32) & 1u) == 0;
                banks |= 1u << (word % 32);
            }
            if (ok) return TiledLayout{pad, x};
        }
    }
    return TiledLayout{~0u, 0};
}

constexpr uint32_t log2_pow2(uint32_t v) { return v <= 1 ? 0 : 1 + log2_pow2(v >> 1); }

// Geometry of the power-of-two tiled gather: element size E, stride S, input
// span per block, threads per block.
template <int E, int S, int kSpanBytes = kTiledPow2SpanBytes, int kThreads = kTiledPow2Threads>
struct TiledPow2 {
    static_assert(S >= 2 && S <= 64 && (S & (S - 1)) == 0, "power-of-two stride from 2 to 64");
    static constexpr uint32_t kPerVec = 16 / E;                    // elements per 16-byte load
    static constexpr uint32_t kSpan = kSpanBytes / E;              // input elements per block
    static constexpr uint32_t kP = kSpan / S;                      // positions per lap per block
    static constexpr uint32_t kLog2S = log2_pow2(S);
    static constexpr uint32_t kLoads = kSpan / kPerVec / kThreads;  // 16-byte loads per thread
    static constexpr uint32_t kColStep = kThreads * kPerVec / S;    // columns between a thread's loads
    static constexpr uint32_t kPad = tiled_pow2_layout<E, S, kSpanBytes>().pad;
    static constexpr uint32_t kX = tiled_pow2_layout<E, S, kSpanBytes>().x;
    static constexpr uint32_t kPitch = kP + kPad;
    static constexpr uint32_t kElems = S * kPitch + kX * ((S - 1) >> 5);
    static constexpr int kSmemBytes = static_cast<int>((kElems * E + 15) / 16 * 16);
    static constexpr uint32_t kWarps = kThreads / 32;
    static constexpr uint32_t kWarpsPerLap = S >= static_cast<int>(kWarps) ? 1 : kWarps / S;
    static constexpr uint32_t kSeg = kP / kWarpsPerLap;            // positions of a run per warp
    static_assert(kPad != ~0u, "no bank-conflict-free row layout");
    static_assert(kLoads >= 1 && kLoads * kThreads * kPerVec == kSpan, "whole 16-byte loads per thread");
    static_assert(kThreads >= S, "one thread per lap computes its geometry");
    static_assert(kSeg % (E == 2 ? 64 : 32) == 0, "whole warp-wide words per run share");
    static_assert(E == 4 || (kPitch % 2 == 0 && kX % 2 == 0), "16-bit rows must start on whole words");
    static_assert(S >= static_cast<int>(kPerVec) || (kPitch * E) % 8 == 0, "packed rows start on 8 bytes");
    __host__ __device__ static constexpr uint32_t row_offset(uint32_t r) { return r * kPitch + kX * (r >> 5); }
};

// The element of row r that a 16-byte load v holds at column slot c (S < V):
// element k = c*S + r of the load.
template <int E, int S>
__device__ __forceinline__ uint32_t load_elem(const Vec<16> &v, uint32_t k) {
    return E == 4 ? v.w[k] : (v.w[k >> 1] >> (16u * (k & 1u))) & 0xffffu;
}

template <int E, int S, int kSpanBytes, int kThreads>
__global__ void __launch_bounds__(kThreads) gather_tiled_pow2_kernel(const GatherArgs g) {
    enter_grid();
    using T = TiledPow2<E, S, kSpanBytes, kThreads>;
    using W = typename std::conditional<E == 4, uint32_t, uint16_t>::type;
    __shared__ __align__(16) W tile[T::kElems];
    __shared__ uint32_t lap_start[S], lap_len[S], lap_row[S];
    W *out = static_cast<W *>(g.out);
    const uint32_t p0 = blockIdx.x * T::kP;
    if (threadIdx.x < S) {  // lap L: first output, length, offset of its source row
        const uint32_t L = threadIdx.x, a0 = L * g.lap_m;
        const uint32_t c0 = (a0 + S - 1) >> T::kLog2S;             // ceil(L*m/S)
        const uint32_t c1 = (a0 + g.lap_m + S - 1) >> T::kLog2S;
        lap_start[L] = L * g.lap_q + c0;
        lap_len[L] = g.lap_q + (c1 - c0);
        lap_row[L] = T::row_offset(c0 * S - a0);
    }
    const uint64_t j0 = static_cast<uint64_t>(S) * p0;  // first source of the span
    const W *src = static_cast<const W *>(g.in) + j0;
    const bool full = j0 + T::kSpan <= g.n;              // block-uniform
    if (full) {
        const char *src_bytes = reinterpret_cast<const char *>(src);
        Vec<16> v[T::kLoads];
#pragma unroll
        for (uint32_t i = 0; i < T::kLoads; ++i) v[i] = ld<16>(src_bytes + (threadIdx.x + i * kThreads) * 16u);
        const uint32_t j = T::kPerVec * threadIdx.x;
        if constexpr (S >= static_cast<int>(T::kPerVec)) {  // element k to row (j mod S) + k
            W *dst = tile + T::row_offset(j & (S - 1)) + (j >> T::kLog2S);
#pragma unroll
            for (uint32_t i = 0; i < T::kLoads; ++i) {
#pragma unroll
                for (uint32_t k = 0; k < T::kPerVec; ++k) {
                    const uint32_t w = v[i].w[k * E / 4];
                    dst[k * T::kPitch + i * T::kColStep] = static_cast<W>(E == 4 ? w : w >> (16u * (k & 1u)));
                }
            }
        } else {  // j mod S = 0: element k to row k mod S, column j/S + k/S; V/S columns per row
            constexpr uint32_t kPerRow = T::kPerVec / S;  // 2 or 4 elements: 4 or 8 bytes
            W *dst = tile + (j >> T::kLog2S);
#pragma unroll
            for (uint32_t i = 0; i < T::kLoads; ++i) {
#pragma unroll
                for (uint32_t r = 0; r < static_cast<uint32_t>(S); ++r) {
                    W *at = dst + T::row_offset(r) + i * T::kColStep;
                    uint32_t e[kPerRow];
#pragma unroll
                    for (uint32_t c = 0; c < kPerRow; ++c) e[c] = load_elem<E, S>(v[i], c * S + r);
                    if constexpr (E == 4) {
                        *reinterpret_cast<uint2 *>(at) = make_uint2(e[0], e[1]);
                    } else if constexpr (kPerRow == 2) {
                        *reinterpret_cast<uint32_t *>(at) = e[0] | (e[1] << 16);
                    } else {
                        *reinterpret_cast<uint2 *>(at) = make_uint2(e[0] | (e[1] << 16), e[2] | (e[3] << 16));
                    }
                }
            }
        }
    } else {
        const uint32_t avail = static_cast<uint32_t>(g.n - j0);  // fewer than kSpan
        for (uint32_t j = threadIdx.x; j < avail; j += kThreads)
            tile[T::row_offset(j & (S - 1)) + (j >> T::kLog2S)] = src[j];
    }
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u;
    // work item = (lap, share of its run); one per warp at a time
    for (uint32_t item = threadIdx.x >> 5; item < S * T::kWarpsPerLap; item += T::kWarps) {
        const uint32_t L = item / T::kWarpsPerLap, q0 = (item % T::kWarpsPerLap) * T::kSeg;
        const W *row = tile + lap_row[L] + q0;
        W *dst = out + (static_cast<size_t>(lap_start[L]) + p0 + q0);
        if (full) {  // the whole run [0, P) of every lap lies before n
            if (E == 4 || (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                const uint32_t *row_w = reinterpret_cast<const uint32_t *>(row);
                uint32_t *dst_w = reinterpret_cast<uint32_t *>(dst);
#pragma unroll
                for (uint32_t i = 0; i < T::kSeg * E / 4 / 32; ++i) dst_w[lane + 32 * i] = row_w[lane + 32 * i];
            } else {
#pragma unroll 8
                for (uint32_t i = 0; i < T::kSeg / 32; ++i) dst[lane + 32 * i] = row[lane + 32 * i];
            }
        } else {
            const uint32_t len = lap_len[L] > p0 ? min(lap_len[L] - p0, T::kP) : 0u;
            const uint32_t end = len > q0 ? min(len - q0, T::kSeg) : 0u;
            for (uint32_t q = lane; q < end; q += 32) dst[q] = row[q];
        }
    }
}

template <int E, int S, int kSpanBytes, int kThreads>
cudaError_t launch_gather_tiled_pow2(const GatherArgs &g, int grid, cudaStream_t s) {
    return launch_kernel(&gather_tiled_pow2_kernel<E, S, kSpanBytes, kThreads>, grid, kThreads, 0, s, g);
}

template <int E, int S, int kSpanBytes = kTiledPow2SpanBytes, int kThreads = kTiledPow2Threads>
constexpr GatherEntry tiled_pow2_entry() {
    using T = TiledPow2<E, S, kSpanBytes, kThreads>;
    return GatherEntry{reinterpret_cast<const void *>(&gather_tiled_pow2_kernel<E, S, kSpanBytes, kThreads>),
                       &launch_gather_tiled_pow2<E, S, kSpanBytes, kThreads>, static_cast<int>(T::kLoads),
                       T::kSmemBytes};
}

// Grid-stride gather for any n: with i = v + k*T (T = grid threads),
// (s*i) mod n advances by (s*T) mod n per slot, so each thread needs one
// modular product and then conditional subtractions.
template <int E, int U>
__global__ void __launch_bounds__(kBlock) gather_stride_kernel(const GatherArgs g) {
    enter_grid();
    const char *in = static_cast<const char *>(g.in);
    char *out = static_cast<char *>(g.out);
    const uint64_t n = g.n;
    const uint64_t nthr = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    uint64_t v = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (v >= n) return;
    uint64_t jv = mulmod_u64(g.s_mod, v, n);  // (s*v) mod n, v < n
    for (; v + (U - 1) * nthr < n; v += U * nthr) {
        Vec<E> x[U];
        uint64_t j = jv;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            x[k] = ld<E>(in + j * E);
            j = addmod_u64(j, g.step_mod, n);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) st<E>(out + (v + k * nthr) * E, x[k]);
        jv = j;  // U slots further on: (s*(v + U*T)) mod n
    }
    for (; v < n; v += nthr) {
        st<E>(out + v * E, ld<E>(in + jv * E));
        jv = addmod_u64(jv, g.step_mod, n);
    }
}

// Span gather for a small stride S (2 or 4) on 4-byte elements.  A thread
// owns 8 consecutive outputs i0..i0+7 (one 32-byte store); their sources
// (S*i0 + S*k) mod n lie in the contiguous span j0 .. j0 + 8S - 1 unless the
// span wraps past n.  When it does not wrap and starts 32-byte aligned, the
// thread loads the span with S 256-bit loads and keeps every S-th word (the
// same DRAM sectors as one load per output, an eighth of the load
// instructions); otherwise it falls back to one load per output.
template <int S, int U>
__global__ void __launch_bounds__(kBlock) gather_span_kernel(const GatherArgs g) {
    enter_grid();
    const char *in = static_cast<const char *>(g.in);
    char *out = static_cast<char *>(g.out);
    const uint64_t n = g.n;
    if (blockIdx.x == 0) {  // outputs before 32-byte alignment and after the last vector
        const uint64_t t = threadIdx.x;
        if (t < static_cast<uint64_t>(g.head)) {
            const uint64_t x = g.s_mod * t;
            uint64_t j = x - __umul64hi(x, g.barrett_m) * n;
            j = (j >= n) ? j - n : j;
            j = (j >= n) ? j - n : j;
            st<4>(out + t * 4, ld<4>(in + j * 4));
        }
        if (t < n - static_cast<uint64_t>(g.tail0)) {
            const uint64_t i = static_cast<uint64_t>(g.tail0) + t;
            const uint64_t x = g.s_mod * i;
            uint64_t j = x - __umul64hi(x, g.barrett_m) * n;
            j = (j >= n) ? j - n : j;
            j = (j >= n) ? j - n : j;
            st<4>(out + i * 4, ld<4>(in + j * 4));
        }
    }
    constexpr int64_t kChunk = static_cast<int64_t>(kBlock) * U;  // vectors per chunk
    const int64_t nchunks = (g.nvec + kChunk - 1) / kChunk;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = c * kChunk + threadIdx.x + u * kBlock;
            if (v >= g.nvec) continue;
            const uint64_t i0 = static_cast<uint64_t>(g.head) + 8u * static_cast<uint64_t>(v);
            const uint64_t x = g.s_mod * i0;  // s_mod = S < n <= 2^32
            uint64_t j0 = x - __umul64hi(x, g.barrett_m) * n;
            j0 = (j0 >= n) ? j0 - n : j0;
            j0 = (j0 >= n) ? j0 - n : j0;
            Vec<32> r;
            const char *src = in + j0 * 4;
            if (j0 + 8u * S <= n && (reinterpret_cast<uintptr_t>(src) & 31u) == 0) {
                Vec<32> span[S];
#pragma unroll
                for (int q = 0; q < S; ++q) span[q] = ld<32>(src + q * 32);
#pragma unroll
                for (int k = 0; k < 8; ++k) r.w[k] = span[(k * S) / 8].w[(k * S) % 8];
            } else {
                uint64_t j = j0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    r.w[k] = ld<4>(in + j * 4).w[0];
                    j = addmod_u64(j, static_cast<uint64_t>(S), n);
                }
            }
            st<32>(out + i0 * 4, r);
        }
    }
}

template <int S, int U>
cudaError_t launch_gather_span(const GatherArgs &g, int grid, cudaStream_t s) {
    return launch_kernel(&gather_span_kernel<S, U>, grid, kBlock, 0, s, g);
}

template <int E, int U>
cudaError_t launch_gather_oneshot(const GatherArgs &g, int grid, cudaStream_t s) {
    return launch_kernel(&gather_oneshot_kernel<E, U>, grid, kBlock, 0, s, g);
}
template <int E, int U>
cudaError_t launch_gather_laps(const GatherArgs &g, int grid, cudaStream_t s) {
    return launch_kernel(&gather_laps_kernel<E, U>, grid, kBlock, 0, s, g);
}
template <int E, int U>
cudaError_t launch_gather_tiled(const GatherArgs &g, int grid, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(g.s_mod) * g.tile_pitch * E;
    return launch_kernel(&gather_tiled_kernel<E, U>, grid, kBlock, smem, s, g);
}
template <int E, int U>
cudaError_t launch_gather_stride(const GatherArgs &g, int grid, cudaStream_t s) {
    return launch_kernel(&gather_stride_kernel<E, U>, grid, kBlock, 0, s, g);
}

}  // namespace ew

namespace ew {

// ---------------------------------------------------------------- fixed-stride tiled gather
//
// The tiled schedule for a stride S that is not a power of two but is known
// at compile time.  A thread's 16-byte loads stay in the same rows when the
// block's threads T are chosen so that V*T (V elements per load) is a
// multiple of S: load i of thread t holds span elements V*t + V*T*i + k,
// whose row (V*t + k) mod S does not depend on i and whose column advances
// by V*T/S per load.  So each thread works out, once, the shared-memory
// offset of each of its V elements, and every load's elements go to those
// offsets plus a compile-time step.  T is the smallest multiple of
// lcm(32, S / gcd(S, V)) from 192 threads (384 from S = 32) when that is at
// most 512; otherwise a multiple of S / gcd(S, V) with a partial last warp.
// A block stages about 16 KiB of input (20 KiB for blocks of 352 threads or
// more, 32 KiB from S = 32 so that lap runs stay long; the span is
// kLoads*V*T elements, P = span / S positions per lap).
// The row pitch comes from the host (tile_pitch), chosen for the bank spread
// of these stores; the rows live in dynamic shared memory.  The store phase
// is the power-of-two kernel's: warps share out the lap runs.

constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }
constexpr int lcm_int(int a, int b) { return a / gcd_int(a, b) * b; }

template <int E, int S>
struct TiledFixed {
    static constexpr int kPerVec = 16 / E;
    // A thread's rows stay fixed across its loads when V*T is a multiple of
    // S, i.e. when T is a multiple of kRowPeriod.
    static constexpr int kRowPeriod = S / gcd_int(S, kPerVec);
    // wide strides: bigger blocks and spans, so that lap runs stay long
    static constexpr int kMinThreads = S >= 32 ? 384 : 192;
    static constexpr int kRunAlign = E == 2 ? 64 : 32;
    // Span per block: 16 KiB for blocks of up to 320 threads (6 to 10 per
    // SM), 20 KiB for 352 to 448 threads (4 or 5 per SM), 24 KiB for 480,
    // 32 KiB for the wide strides.  Measured on GB300 at 2^26: 224- and
    // 288-thread blocks staging 17.5-18 KiB instead of 14-13.5 lost 3-8% on
    // 16-bit elements (the shared memory then crowds out the L1 the loads in
    // flight use), while 352- and 416-thread blocks staging 16.5-19.5 KiB
    // instead of 11-13 gained 4-7% (s = 11, 13, 22, 26) on both element
    // sizes, and 480-thread blocks (s = 15, 30) 22.5 KiB instead of 15 gained
    // 3-5% (7% on an input past a 16-byte boundary).
    static constexpr int target_bytes(int t) {
        return S >= 32 ? 32768 : t >= 480 ? 24576 : t >= 352 ? 20480 : 16384;
    }
    static constexpr int warps_per_lap(int t) { return S >= t / 32 ? 1 : (t / 32) / S; }
    // loads per thread: from about target_bytes of span up, the first count
    // that gives each warp's share of a run a whole number of warp-wide
    // 4-byte words (-1 if none up to 64)
    static constexpr int loads_from(int t, int l) {
        return l > 64 ? -1
                      : (l * kPerVec * t / S) % (kRunAlign * warps_per_lap(t)) == 0 ? l : loads_from(t, l + 1);
    }
    static constexpr int loads_for(int t) {
        return loads_from(t, target_bytes(t) / (16 * t) > 0 ? target_bytes(t) / (16 * t) : 1);
    }
    // Threads: the smallest multiple of lcm(32, kRowPeriod) from kMinThreads
    // (whole warps), if that is at most 512.  Otherwise (odd strides from 17,
    // and 34-62 where 4 or 8 does not divide them) a multiple of kRowPeriod
    // up to 512 whose span comes nearest its target, whole warps breaking
    // ties; the last warp is then partial and takes part in the staging only.
    static constexpr int kWholeWarps = (kMinThreads + lcm_int(32, kRowPeriod) - 1) / lcm_int(32, kRowPeriod) *
                                       lcm_int(32, kRowPeriod);
    static constexpr int deviation(int t) {
        return loads_for(t) < 0 ? 1 << 30
                                : (loads_for(t) * 16 * t > target_bytes(t) ? loads_for(t) * 16 * t - target_bytes(t)
                                                                            : target_bytes(t) - loads_for(t) * 16 * t);
    }
    static constexpr int pick_threads() {
        if (kWholeWarps <= 512) return kWholeWarps;
        int best = 0;
        for (int t = (kMinThreads + kRowPeriod - 1) / kRowPeriod * kRowPeriod; t <= 512; t += kRowPeriod) {
            if (best == 0 || deviation(t) < deviation(best) ||
                (deviation(t) == deviation(best) && t % 32 == 0 && best % 32 != 0))
                best = t;
        }
        return best;
    }
    static constexpr int kThreads = pick_threads();
    static constexpr int kWarps = kThreads / 32;  // whole warps: the store phase
    // 192- and 384-thread blocks (s = 3, 6, 12, 24, 48) ask for at least one
    // resident block per SM, which lets the compiler use more registers (40-44
    // for 16-bit elements) than the 32 that keep 2048 threads resident.
    // Measured on GB300 at 2^26 over every stride from 3 to 63, two rounds:
    // those five strides gained 1-6% for 16-bit elements and 0.2-1.1% for
    // fp32, while the other blocks of whole warps lost up to 4.6% (16-bit)
    // and the partial-warp ones up to 4%, so the rest keep the default (0).
    static constexpr int kMinBlocks = kThreads == 192 || kThreads == 384 ? 1 : 0;
    static constexpr int kWarpsPerLap = warps_per_lap(kThreads);
    static constexpr int kLoads = loads_for(kThreads);
    static constexpr int kSpan = kLoads * kPerVec * kThreads;  // elements
    static constexpr int kP = kSpan / S;
    static constexpr int kColStep = kPerVec * kThreads / S;
    static constexpr int kSeg = kP / kWarpsPerLap;
    static constexpr int kWraps = (kPerVec - 1) / S + 1;  // row wraps within one load, at most
    static_assert(kThreads <= 512 && kThreads >= S && kWarps >= 1, "block size");
    static_assert(kLoads >= 1 && deviation(kThreads) < (1 << 30), "span");
    static_assert((kPerVec * kThreads) % S == 0 && kSpan % S == 0, "rows invariant across a thread's loads");
    static_assert(kSeg % kRunAlign == 0, "whole warp-wide words per run share");
};

template <int E, int S, bool kShifted>
__global__ void __launch_bounds__(TiledFixed<E, S>::kThreads, TiledFixed<E, S>::kMinBlocks)
gather_tiled_fixed_kernel(const GatherArgs g) {
    enter_grid();
    using T = TiledFixed<E, S>;
    using W = typename std::conditional<E == 4, uint32_t, uint16_t>::type;
    extern __shared__ __align__(16) unsigned char fixed_raw[];
    W *tile = reinterpret_cast<W *>(fixed_raw);
    __shared__ uint32_t lap_start[S], lap_len[S], lap_row[S];
    const uint32_t pitch = g.tile_pitch;
    W *out = static_cast<W *>(g.out);
    const uint32_t p0 = blockIdx.x * static_cast<uint32_t>(T::kP);
    if (threadIdx.x < S) {  // lap L: first output, length, offset of its source row
        const uint32_t L = threadIdx.x, a0 = L * g.lap_m;
        const uint32_t c0 = (a0 + S - 1) / S;                  // ceil(L*m/S)
        const uint32_t c1 = (a0 + g.lap_m + S - 1) / S;
        lap_start[L] = L * g.lap_q + c0;
        lap_len[L] = g.lap_q + (c1 - c0);
        lap_row[L] = (c0 * S - a0) * pitch;
    }
    const uint64_t j0 = static_cast<uint64_t>(S) * p0;  // first source of the span
    const W *src = static_cast<const W *>(g.in) + j0;
    const bool full = j0 + T::kSpan <= g.n;              // block-uniform
    // An input d elements past a 16-byte boundary (the kShifted instances):
    // every span starts d elements past one too (a span is a whole number of
    // 16-byte loads), so the loads are shifted back by d.  Load i of thread t
    // then holds span elements V*(t + T*i) + k - d, still in rows fixed
    // across i.  Thread 0's first load would start before the span and is
    // skipped; the V elements not covered (the valid part of that load and
    // the span's last d) are staged singly.  The aligned instances compile
    // with d = 0, without that work.
    const uint32_t d = kShifted ? (static_cast<uint32_t>(reinterpret_cast<uintptr_t>(g.in)) & 15u) / E : 0u;
    if (full) {
        const char *src_bytes = reinterpret_cast<const char *>(src) - d * E;
        Vec<16> v[T::kLoads];
#pragma unroll
        for (int i = 0; i < T::kLoads; ++i)
            if (!kShifted || i > 0 || d == 0 || threadIdx.x > 0)
                v[i] = ld<16>(src_bytes + (threadIdx.x + i * T::kThreads) * 16u);
        // span elements [0, V - d) and [span - d, span), staged singly: loaded
        // here, with the vector loads, so that their latency overlaps
        const bool single = kShifted && d != 0 && threadIdx.x < T::kPerVec;
        const uint32_t single_j =
            threadIdx.x < T::kPerVec - d ? threadIdx.x : T::kSpan - T::kPerVec + threadIdx.x;
        W single_v = 0;
        if (single) single_v = src[single_j];
        // offsets of this thread's V elements in its first load (rows fixed
        // across its loads)
        uint32_t at[T::kPerVec];
        if constexpr (kShifted) {
            // from span index V*t + k - d, made non-negative by adding V*S.
            // For thread 0 with d > 0 the first columns are -1 or less: the
            // offset wraps modulo 2^32, and only that thread's later loads
            // use it, whose columns (+ i*kColStep) are back at 0 or more
#pragma unroll
            for (int k = 0; k < T::kPerVec; ++k) {
                const uint32_t jp = T::kPerVec * threadIdx.x + k - d + T::kPerVec * S;
                at[k] = (jp % S) * pitch + jp / S - T::kPerVec;
            }
        } else {
            const uint32_t j = T::kPerVec * threadIdx.x;
            const uint32_t r0 = j % S, c0 = j / S;
#pragma unroll
            for (int k = 0; k < T::kPerVec; ++k) {
                uint32_t r = r0 + k, c = c0;
#pragma unroll
                for (int w = 0; w < T::kWraps; ++w) {
                    const bool wrap = r >= S;
                    r = wrap ? r - S : r;
                    c = wrap ? c + 1 : c;
                }
                at[k] = r * pitch + c;
            }
        }
#pragma unroll
        for (int i = 0; i < T::kLoads; ++i) {
            if (kShifted && i == 0 && d != 0 && threadIdx.x == 0) continue;
#pragma unroll
            for (int k = 0; k < T::kPerVec; ++k) {
                const uint32_t w = v[i].w[k * E / 4];
                tile[at[k] + i * T::kColStep] = static_cast<W>(E == 4 ? w : w >> (16u * (k & 1)));
            }
        }
        if (single) tile[(single_j % S) * pitch + single_j / S] = single_v;
    } else {
        const uint32_t avail = static_cast<uint32_t>(g.n - j0);  // fewer than kSpan
        for (uint32_t j = threadIdx.x; j < avail; j += T::kThreads) tile[(j % S) * pitch + j / S] = src[j];
    }
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u;
    // whole warps only: a partial last warp (T not a multiple of 32) has
    // done its share in the staging
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t items = static_cast<uint32_t>(S * T::kWarpsPerLap);
    for (uint32_t item = warp; warp < T::kWarps && item < items; item += T::kWarps) {
        const uint32_t L = item / T::kWarpsPerLap, q0 = (item % T::kWarpsPerLap) * T::kSeg;
        const W *row = tile + lap_row[L] + q0;
        W *dst = out + (static_cast<size_t>(lap_start[L]) + p0 + q0);
        if (full) {
            if (E == 4 || (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                const uint32_t *row_w = reinterpret_cast<const uint32_t *>(row);
                uint32_t *dst_w = reinterpret_cast<uint32_t *>(dst);
#pragma unroll 8
                for (int i = 0; i < T::kSeg * E / 4 / 32; ++i) dst_w[lane + 32 * i] = row_w[lane + 32 * i];
            } else {
#pragma unroll 8
                for (int i = 0; i < T::kSeg / 32; ++i) dst[lane + 32 * i] = row[lane + 32 * i];
            }
        } else {
            const uint32_t len = lap_len[L] > p0 ? min(lap_len[L] - p0, static_cast<uint32_t>(T::kP)) : 0u;
            const uint32_t end = len > q0 ? min(len - q0, static_cast<uint32_t>(T::kSeg)) : 0u;
            for (uint32_t q = lane; q < end; q += 32) dst[q] = row[q];
        }
    }
}

template <int E, int S, bool kShifted>
cudaError_t launch_gather_tiled_fixed(const GatherArgs &g, int grid, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(S) * g.tile_pitch * E;
    return launch_kernel(&gather_tiled_fixed_kernel<E, S, kShifted>, grid, TiledFixed<E, S>::kThreads, smem, s, g);
}

template <int E, int S, bool kShifted>
constexpr GatherEntry tiled_fixed_entry() {
    using T = TiledFixed<E, S>;
    return GatherEntry{reinterpret_cast<const void *>(&gather_tiled_fixed_kernel<E, S, kShifted>),
                       &launch_gather_tiled_fixed<E, S, kShifted>, T::kLoads, 0, T::kThreads,
                       static_cast<uint32_t>(T::kP)};
}

}  // namespace ew
