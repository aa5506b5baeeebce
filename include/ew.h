/*
 * ew.h -- C ABI of libew.so, memory-bound elementwise operators for GB300
 * (sm_103a).
 *
 * Operations (each output element depends only on the same index of the
 * inputs, "逐元素操作算子" §一.1, except the gather):
 *
 *   ew_add            C[i] = A[i] + B[i]
 *                     "HyperAI elementwise add on RTX 5090" (hyper.ai), Versions
 *                     1-6; "逐元素操作算子" §二 template kernel.
 *   ew_saxpy          y[i] = alpha * x[i] + y[i], in place, one fused multiply-add
 *                     "Puzzle 31: occupancy optimisation" (puzzles.modular.com),
 *                     overview and minimal kernel.
 *   ew_relu           y[i] = max(x[i], 0)
 *                     CUDA-MODE lecture notes (cyqw.cn/news/898472), §5.2 example 1.
 *   ew_add_relu       C[i] = max(A[i] + B[i], 0) in one pass
 *                     CUDA-MODE lecture notes, §5.3 (kernel fusion).
 *   ew_saxpy_relu     y[i] = max(alpha * x[i] + y[i], 0), in place, in one pass
 *                     CUDA-MODE lecture notes, §5.3 (kernel fusion).
 *   ew_select_even_odd y[i] = x[i] even ? 2 x[i] : x[i] + 1 on 32-bit integers
 *                     CUDA-MODE lecture notes, §6.1-6.2 (control divergence).
 *   ew_copy           out[i] = in[i]
 *                     CUDA-MODE lecture notes, §3.2 coalesced version.
 *   ew_gather_stride  out[i] = in[(stride * i) mod n]
 *                     CUDA-MODE lecture notes, §3.2 non-coalesced version (stride 2).
 *
 * Arithmetic (bit-exact, no tolerance):
 *   f32 add      IEEE binary32 addition, round to nearest even; subnormals kept.
 *   f16/bf16 add the exact sum rounded once to the format, nearest even.  This
 *                equals "binary32 add, then one rounding" (binary32 carries more
 *                than 2p+1 significand bits for both formats).
 *   saxpy        f32: fmaf(alpha, x, y), one rounding.  f16/bf16: x and y widened
 *                exactly to binary32, fmaf there, then one rounding to the format.
 *                alpha is binary32 and is never rounded to the 16-bit format.
 *   relu         x > 0 -> x;  x <= 0 (including -0) -> +0;  NaN -> x unchanged.
 *   add_relu     relu applied to the rounded sum of add.
 *   saxpy_relu   relu applied to the rounded result of saxpy.
 *   select       two's complement int32, wrapping modulo 2^32.
 *   copy/gather  raw element bits.
 *
 * Common conventions
 *   Pointers   any memory the current device can address, owned by the caller:
 *              device memory (cudaMalloc, cudaMallocAsync), managed memory,
 *              page-locked host memory, and on devices with pageable memory
 *              access (GB300 with its Grace CPU) plain host memory too, which
 *              the kernels then read and write over the CPU-GPU link.  The library
 *              allocates no memory and keeps no reference after a call returns.
 *              Each pointer must be aligned to the element size (4 bytes for
 *              EW_F32 and EW_I32, 2 for EW_F16/EW_BF16), else
 *              EW_ERR_INVALID_VALUE.  Any such alignment is accepted; the
 *              widest vector width that all the pointers of a call share is
 *              used, or, for 16-bit pointers of different parity from
 *              n = 2^22 on device memory, the realigning bulk copy (see
 *              EW_PATH_TMA and ew_plan_query).
 *   Layout     n contiguous elements, index 0 first.
 *   n          element count.  n == 0 returns EW_OK and launches nothing;
 *              n < 0 is EW_ERR_INVALID_VALUE.
 *   Aliasing   an output may be *identical* to an input (in-place add, saxpy
 *              and saxpy_relu with x == y, relu, copy).  Any other overlap of an output's byte
 *              range with an input's is EW_ERR_OVERLAP.  ew_gather_stride
 *              accepts no overlap at all.
 *   Streams    every call enqueues at most one kernel on `stream` (NULL = the
 *              legacy default stream) on the calling thread's current device and
 *              returns without synchronising.  Kernels are launched with
 *              programmatic dependent launch unless ew_set_programmatic_launch(0)
 *              (see there).  Device faults surface at the caller's next
 *              synchronisation.
 *   Errors     every call returns an ew_status and never prints or aborts.
 *              Argument errors are detected on the host before any CUDA call.
 *              EW_ERR_CUDA: a CUDA runtime call or the launch failed; the
 *              cudaError_t value is kept per thread (ew_last_cuda_error).
 *   Threads    all entry points are thread-safe.  The variant selections
 *              (ew_set_path, ew_set_schedule, ew_set_programmatic_launch,
 *              ew_set_pointer_check) are process-wide.
 */
#ifndef EW_H
#define EW_H

#include <stdint.h>

#if defined(__GNUC__)
#define EW_API __attribute__((visibility("default")))
#else
#define EW_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *), so no CUDA header is needed. */
typedef struct CUstream_st *ew_stream_t;

typedef enum {
    EW_F32 = 0,  /* IEEE binary32 */
    EW_F16 = 1,  /* IEEE binary16 */
    EW_BF16 = 2, /* bfloat16 (upper half of binary32) */
    EW_I32 = 3   /* 32-bit two's complement integer: ew_select_even_odd, ew_copy and
                    ew_gather_stride only (others return EW_ERR_UNSUPPORTED_DTYPE) */
} ew_dtype;

typedef enum {
    EW_OK = 0,
    EW_ERR_INVALID_VALUE = 1,     /* n < 0, stride <= 0, misaligned pointer, bad enum */
    EW_ERR_NULL_POINTER = 2,      /* a NULL pointer with n > 0 */
    EW_ERR_UNSUPPORTED_DTYPE = 3, /* dtype outside ew_dtype, or not one the operation takes */
    EW_ERR_OVERLAP = 4,           /* partial overlap between an input and the output */
    EW_ERR_NOT_DEVICE_POINTER = 5,/* pointer check enabled and a pointer is not device-accessible */
    EW_ERR_CUDA = 6,              /* CUDA runtime error; see ew_last_cuda_error */
    EW_ERR_TIMEOUT = 7            /* a bounded device-side wait gave up (see ew_device_error) */
} ew_status;

/* Kernel variant for the body of a call.  EW_PATH_AUTO picks the fastest
 * measured variant that the pointers' alignment allows: the widest access
 * width all the pointers share, up to 32 bytes. */
typedef enum {
    EW_PATH_AUTO = 0,
    EW_PATH_SCALAR = 1, /* one element per access, grid-stride */
    EW_PATH_V128 = 2,   /* 16-byte vector accesses */
    EW_PATH_V256 = 3,   /* 32-byte vector accesses (sm_100 family) */
    EW_PATH_TMA = 4     /* bulk async copies (cp.async.bulk) through shared memory,
                           for device memory.  Pointers that disagree modulo 16
                           bytes take a realigning kernel: each input tile is
                           copied as the 16-byte aligned span around it and read
                           at its offset in shared memory.  EW_PATH_AUTO uses
                           that kernel for 16-bit elements whose pointers differ
                           in parity (2-byte accesses otherwise) from n >= 2^22,
                           after checking that every pointer is device memory;
                           during stream capture it keeps the vector kernel */
} ew_path;

/* How the body's chunks are handed to thread blocks.
 * EW_SCHED_ONESHOT    one block per chunk of 256 threads x 64 bytes per thread
 *                     per input; the hardware block scheduler balances the SMs
 *                     (the default: fastest measured on GB300).  The gather
 *                     walks its outputs in index order.
 * EW_SCHED_PERSISTENT at most SMs x resident blocks per SM, each striding over
 *                     the chunks (the grid-stride design of the pages).
 * EW_SCHED_LAPS       gather only (the other operators run EW_SCHED_ONESHOT):
 *                     as i runs over the outputs, (stride * i) mod n sweeps the
 *                     input s = (stride mod n) times.  One block per chunk of
 *                     2048 outputs of one sweep ("lap"), with the s laps'
 *                     blocks interleaved so that the blocks running together
 *                     read the same stretch of the input and each sector comes
 *                     from DRAM once.  It applies when 2 <= s <= 64,
 *                     n <= 2^32 and n >= 2048 s; otherwise EW_SCHED_ONESHOT
 *                     runs.
 * EW_SCHED_TILED      gather only, same range of s and n as EW_SCHED_LAPS (any
 *                     n >= 1 there): the transpose-like schedule.  A block
 *                     reads the contiguous input span that its positions of
 *                     all s laps draw from (12-32 KiB) once, coalesced, into
 *                     shared memory with one row per residue mod s, then
 *                     writes each lap's outputs as one coalesced run.  For
 *                     every s from 2 to 64 on an input aligned to 16 bytes,
 *                     and for the s that are not powers of two (and, for
 *                     2-byte elements, s = 2, 4, 8) on any input, a kernel
 *                     specialised for that stride runs
 *                     (division by s at compile time, staging stores at
 *                     fixed offsets, a padded shared-memory layout, warps
 *                     copying whole lap runs; the launch record shows
 *                     EW_PATH_V128 and the block size chosen for the
 *                     stride).
 * EW_SCHED_AUTO       for the gather: EW_SCHED_LAPS for s < 5, EW_SCHED_TILED
 *                     for 5 <= s <= 64 (the measured crossover: a
 *                     lap-ordered warp load fetches more sectors per useful
 *                     byte as s grows, and 16-bit lanes move 2 bytes each);
 *                     2-byte elements take EW_SCHED_TILED from s = 2.
 *                     For the other operators,
 *                     EW_SCHED_ONESHOT.  A gather with n > 2^32 always runs
 *                     persistent. */
typedef enum {
    EW_SCHED_AUTO = 0,
    EW_SCHED_ONESHOT = 1,
    EW_SCHED_PERSISTENT = 2,
    EW_SCHED_LAPS = 3,
    EW_SCHED_TILED = 4
} ew_schedule;

/* ---- operators ------------------------------------------------------- */

/* C = A + B.  a, b: n input elements; c: n output elements (c may be a or b). */
EW_API ew_status ew_add(ew_dtype dtype, const void *a, const void *b, void *c, int64_t n,
                 ew_stream_t stream);

/* y = alpha * x + y in place.  x: n inputs; y: n inputs overwritten with the
 * result (x == y is allowed). */
EW_API ew_status ew_saxpy(ew_dtype dtype, float alpha, const void *x, void *y, int64_t n,
                   ew_stream_t stream);

/* y = max(x, 0).  x: n inputs; y: n outputs (y == x computes in place).  In
 * place, a vector the operation leaves unchanged (no negative element and no
 * -0) is not written back: CUDA-MODE lecture notes §5.2, example 1, case B,
 * where a non-negative element needs no write. */
EW_API ew_status ew_relu(ew_dtype dtype, const void *x, void *y, int64_t n, ew_stream_t stream);

/* C = max(A + B, 0): the sum rounded as in ew_add, then ReLU as in ew_relu, in
 * one pass over memory (a bias add fused with its activation; kernel fusion as
 * CUDA-MODE lecture notes §5.3 lists it for memory-bound work).  Arguments and
 * aliasing as in ew_add. */
EW_API ew_status ew_add_relu(ew_dtype dtype, const void *a, const void *b, void *c, int64_t n,
                             ew_stream_t stream);

/* y = max(alpha * x + y, 0) in place: the result rounded as in ew_saxpy, then
 * ReLU as in ew_relu, in one pass over memory (CUDA-MODE lecture notes §5.3,
 * kernel fusion).  Arguments and aliasing as in ew_saxpy. */
EW_API ew_status ew_saxpy_relu(ew_dtype dtype, float alpha, const void *x, void *y, int64_t n,
                               ew_stream_t stream);

/* y = x even ? 2x : x + 1, on EW_I32 only, wrapping modulo 2^32: the
 * control-divergence example of CUDA-MODE lecture notes §6.1-6.2 (an if/else
 * on x % 2 and its branch-free rewrite compute the same thing), computed
 * without a branch.  x: n inputs; y: n outputs (y == x computes in place). */
EW_API ew_status ew_select_even_odd(ew_dtype dtype, const void *x, void *y, int64_t n,
                                    ew_stream_t stream);

/* out = in.  in == out is a no-op that launches nothing. */
EW_API ew_status ew_copy(ew_dtype dtype, const void *in, void *out, int64_t n, ew_stream_t stream);

/* out[i] = in[(stride * i) mod n] for i in [0, n); the product is formed
 * without overflow.  stride >= 1 (else EW_ERR_INVALID_VALUE).  in and out must
 * not overlap.  As in the page's non-coalesced copy, each thread reads one
 * element per access, so a warp's load touches every stride-th element of a
 * span while its store covers consecutive elements (except under
 * EW_SCHED_TILED, which stages the input through shared memory).  The order
 * in which blocks take the outputs follows ew_set_schedule.
 * With ew_set_path
 * (EW_PATH_V256) selected, 4-byte elements with (stride mod n) of 2 or 4 and
 * n <= 2^32 use a span variant instead: each thread loads the contiguous
 * source span of 8 outputs with 256-bit loads and keeps every stride-th word
 * (same DRAM sectors, an eighth of the load instructions). */
EW_API ew_status ew_gather_stride(ew_dtype dtype, const void *in, void *out, int64_t n,
                           int64_t stride, ew_stream_t stream);

/* ---- variant selection and introspection ------------------------------ */

/* Select the kernel variant for later calls in this process (EW_PATH_AUTO
 * restores the default).  A forced variant that the alignment of a call does
 * not allow falls back to the widest one it does.  EW_ERR_INVALID_VALUE for a
 * value outside ew_path. */
EW_API ew_status ew_set_path(ew_path path);
EW_API ew_path ew_get_path(void);

/* Select the block schedule for later calls in this process (process-wide).
 * EW_ERR_INVALID_VALUE for a value outside ew_schedule.  The bulk-copy path
 * always runs one-shot. */
EW_API ew_status ew_set_schedule(ew_schedule schedule);
EW_API ew_schedule ew_get_schedule(void);

/* Programmatic dependent launch, enabled (1) by default; 0 disables it.  When
 * enabled, kernels are launched with programmatic stream serialisation: a
 * call's blocks may be scheduled while the previous kernel on the stream is
 * still finishing, and wait (griddepcontrol.wait) for it to complete and its
 * writes to be visible before touching memory.  Results and memory order
 * between calls are the same either way; chains of short calls run faster.
 * Process-wide.  EW_ERR_INVALID_VALUE for other values. */
EW_API ew_status ew_set_programmatic_launch(int enable);
EW_API int ew_get_programmatic_launch(void);

/* Enable (1) or disable (0, the default) a cudaPointerGetAttributes check of
 * every pointer before launch: device, managed and page-locked host memory
 * pass, pageable host memory passes only on a device with pageable memory
 * access; anything else gives EW_ERR_NOT_DEVICE_POINTER.  Process-wide.  The
 * environment variable EW_CHECK_POINTERS=1 enables it at start-up. */
EW_API ew_status ew_set_pointer_check(int enable);

/* How an ew_add / ew_saxpy / ew_relu / ew_add_relu / ew_saxpy_relu / ew_select_even_odd /
 * ew_copy call with these pointers is split under the current ew_set_path
 * selection (host arithmetic only; needs no GPU).  ptrs: the call's input
 * pointers, then its output pointer last; nptrs in [1, 4].  When the pointers
 * disagree modulo 16 bytes, a bulk-copy plan (EW_PATH_TMA, and EW_PATH_AUTO
 * for 16-bit elements of different parity from n >= 2^22, where the call
 * itself also requires device memory) stages each input
 * as the aligned span around its tile: the head then aligns the output only
 * and is at least 16 bytes, and the tail is at least 16 bytes when there is a
 * tile. */
typedef struct {
    int32_t path;      /* ew_path that will run */
    int32_t vec_bytes; /* bytes per access in the body (element size for SCALAR) */
    int64_t head;      /* leading elements done one by one, to reach vector alignment */
    int64_t nvec;      /* whole vectors in the body */
    int64_t tail;      /* trailing elements done one by one */
} ew_plan;
EW_API ew_status ew_plan_query(ew_dtype dtype, const void *const *ptrs, int32_t nptrs, int64_t n,
                        ew_plan *out);

/* What the most recent operator call on this thread launched. */
typedef struct {
    int32_t launches;  /* kernels enqueued by the call (0 or 1) */
    int32_t path;      /* ew_path that ran */
    int32_t vec_bytes;
    int32_t grid;      /* blocks */
    int32_t block;     /* threads per block */
    int32_t smem;      /* dynamic shared memory bytes per block */
    int32_t schedule;  /* ew_schedule that ran */
    int64_t head, nvec, tail; /* for EW_PATH_TMA: nvec counts tiles of 8 KiB per input */
} ew_launch_record;
EW_API ew_status ew_last_launch(ew_launch_record *out);

/* The launch record an ew_gather_stride call with these arguments would leave,
 * under the current ew_set_path / ew_set_schedule selections (host arithmetic
 * only; needs no GPU and reads neither buffer): which kernel schedule, its
 * grid, block, dynamic shared memory and access width.  One exception: the
 * grid of the grid-stride kernel (EW_SCHED_PERSISTENT, or n > 2^32), which
 * depends on the device's SM count and occupancy, is reported as 0.  Returns
 * what ew_gather_stride returns for the same arguments, without its optional
 * pointer-kind check; n == 0 gives a record with launches = 0.  out_record:
 * caller-owned; EW_ERR_NULL_POINTER when null. */
EW_API ew_status ew_gather_plan_query(ew_dtype dtype, const void *in, const void *out, int64_t n,
                                      int64_t stride, ew_launch_record *out_record);

/* ---- errors ----------------------------------------------------------- */

EW_API const char *ew_status_string(ew_status status);

/* cudaError_t value behind the last EW_ERR_CUDA returned on this thread (0 if none). */
EW_API int ew_last_cuda_error(void);

/* Read and clear the device-side error word of the current device, in stream
 * order on `stream`, then synchronise `stream`.  The read and the clear are one
 * atomic exchange on the device: a code that a kernel on another stream records
 * meanwhile is either returned here or kept for the next call.  *code = 0 when
 * no bounded wait has given up since the last read; otherwise the wait site
 * that gave up:
 *   1   a tile of a bulk-copy kernel: under EW_PATH_TMA, and under
 *       EW_PATH_AUTO for 16-bit operands whose pointers differ in parity, from
 *       n >= 2^22 on device memory (the realigning bulk copy).  The outputs of
 *       the calls that ran such a kernel since the last read are undefined:
 *       the CTA that gave up skipped its remaining tiles, and if its second
 *       bounded wait (for loads already issued) also expired it left with
 *       loads still in flight.  Callers of those paths that must know their
 *       results are complete check this word after synchronising.
 *   99  ew_selftest_bounded_wait.
 * Returns EW_ERR_TIMEOUT when *code != 0, EW_ERR_CUDA when the exchange, the
 * copy or the synchronisation fails. */
EW_API ew_status ew_device_error(ew_stream_t stream, int32_t *code);

/* Self-test of the bounded device waits: enqueues one block that arms an
 * mbarrier no copy will complete; its wait must give up after limit_ns
 * nanoseconds (1 <= limit_ns <= 10^10, else EW_ERR_INVALID_VALUE) and record
 * code 99, which a following ew_device_error returns.  Nothing else is touched. */
EW_API ew_status ew_selftest_bounded_wait(int64_t limit_ns, ew_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
EW_API int ew_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EW_H */
