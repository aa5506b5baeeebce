// ew_internal.h -- interface between the host dispatcher (ew_api.cu) and the
// kernel translation units (ew_kernels_*.cu, ew_tma.cu).  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ew {

constexpr int kBlock = 256;  // threads per block for the LSU kernels

// Programmatic dependent launch: when enabled (the default), every kernel is
// launched with programmatic stream serialisation, starts by waiting for the
// grid before it on the stream to complete and flush (griddepcontrol.wait),
// and at once lets the grid after it be scheduled (launch_dependents).  The
// next call's blocks then take SM slots while this call's last blocks drain;
// memory order between calls is unchanged.
bool programmatic_launch();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                          cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (programmatic_launch()) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    // The launch's own status: an error recorded earlier on this thread by
    // another runtime call is not this call's failure and is left alone.
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) (void)cudaGetLastError();  // the failure is returned; do not leave it pending too
    return e;
}

// Operator ids of the streaming (contiguous) kernels.
enum OpId : int {
    OP_ADD = 0, OP_SAXPY = 1, OP_RELU = 2, OP_COPY = 3, OP_ADD_RELU = 4, OP_SELECT = 5, OP_SAXPY_RELU = 6,
    OP_COUNT = 7
};
// Element-size classes of the kernel tables: the 4-byte table serves binary32
// and int32, the 16-bit tables binary16 and bfloat16 (ids match ew_dtype for
// the floating-point types).
enum DtId : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_COUNT = 3 };

// Vector widths in bytes, indexed 0..4 -> 32, 16, 8, 4, 2.
constexpr int kVecBytes[5] = {32, 16, 8, 4, 2};
inline int vec_index(int vb) {
    return vb == 32 ? 0 : vb == 16 ? 1 : vb == 8 ? 2 : vb == 4 ? 3 : 4;
}

// Arguments of one streaming launch.  Elements [0, head) and [tail0, n) are
// done one by one; the body is nvec vectors starting at element head.
struct StreamArgs {
    const void *in0;  // A (add), x (saxpy), x (relu), in (copy)
    const void *in1;  // B (add), y (saxpy); unused otherwise
    void *out;        // C (add), y (saxpy), y (relu), out (copy)
    int64_t n;
    int64_t head;
    int64_t nvec;
    int64_t tail0;
    float alpha;
    int32_t skip_unchanged;  // in-place ReLU: store only vectors whose bits change
};

using StreamLaunchFn = cudaError_t (*)(const StreamArgs &, int grid, cudaStream_t);

struct StreamEntry {
    const void *kernel;     // for occupancy queries
    StreamLaunchFn launch;  // nullptr where the width does not apply
    int unroll;             // vectors in flight per thread per input
};

// Tables filled by the kernel translation units: [op][vec_index].
const StreamEntry *stream_table_f32();   // OP_COUNT x 5
const StreamEntry *stream_table_f16();
const StreamEntry *stream_table_bf16();

// Strided gather: out[i] = in[(s*i) mod n].
struct GatherArgs {
    const void *in;
    void *out;
    uint64_t n;
    uint64_t s_mod;      // stride mod n
    uint64_t step_mod;   // one-shot: (stride * kBlock) mod n; grid-stride: (stride * grid threads) mod n
    uint64_t barrett_m;  // floor((2^64 - 1) / n), one-shot and span kernels
    int64_t head;        // span kernel: outputs [0, head) one by one (32-byte output alignment)
    int64_t nvec;        // span kernel: 8-element output vectors after the head
    int64_t tail0;       // span kernel: outputs [tail0, n) one by one
    uint32_t lap_q;      // lap kernel: n / s_mod
    uint32_t lap_m;      // lap kernel: n mod s_mod
    uint32_t div_magic;  // lap and tiled kernels: floor(2^32 / s_mod) + 1
    uint32_t tile_p;     // tiled kernel: lap positions per block (a power of two)
    uint32_t tile_pitch; // elements per shared-memory row (tile_p plus bank padding)
};
using GatherLaunchFn = cudaError_t (*)(const GatherArgs &, int grid, cudaStream_t);
struct GatherEntry {
    const void *kernel;
    GatherLaunchFn launch;
    int unroll;
    int smem_bytes = 0;  // static shared memory per block, for the launch record
    int block = kBlock;  // threads per block
    uint32_t tile_p = 0; // lap positions per block of the fixed-stride tiled kernels
};
// Lap-ordered gather: 2 <= s_mod <= kMaxLaps, n <= 2^32 and n >= s_mod x the
// outputs of one block.
constexpr uint64_t kMaxLaps = 64;
const GatherEntry *gather_laps_4();
const GatherEntry *gather_laps_2();
// Tiled (transposing) gather: same range as the lap kernel; a block stages
// at most kTiledStageBytes of input in shared memory (more when that would
// leave lap runs shorter than kTiledMinRunBytes).
constexpr uint32_t kTiledStageBytes = 20480;
constexpr uint32_t kTiledMinRunBytes = 512;
const GatherEntry *gather_tiled_4();
const GatherEntry *gather_tiled_2();
// Tiled gather specialised for a power-of-two stride (2, 4, ..., 64) and an
// input aligned to 16 bytes; nullptr for other strides.  Each block of
// kTiledPow2Threads threads stages kTiledPow2SpanBytes of input.
constexpr int kTiledPow2SpanBytes = 16384;
constexpr int kTiledPow2Threads = 256;
const GatherEntry *gather_tiled_pow2_4(uint64_t stride);
const GatherEntry *gather_tiled_pow2_2(uint64_t stride);
// Tiled gather specialised for a fixed stride that is not a power of two
// (every stride from 3 to 63 but 4, 8, 16, 32), on any element-aligned
// input; shifted selects the instance for an input that is not 16-byte
// aligned, which also exists for 2-byte elements at s = 2, 4 and 8.  The block
// size is chosen per stride, the row pitch (args.tile_pitch) by the host.
// nullptr for other strides.
const GatherEntry *gather_tiled_fixed(int e, uint64_t stride, bool shifted);
const GatherEntry *gather_tiled_fixed_wide(int e, uint64_t stride, bool shifted);  // strides 33 to 63
const GatherEntry *gather_oneshot_4();  // binary32, n <= 2^32
const GatherEntry *gather_stride_4();   // binary32, any n
const GatherEntry *gather_oneshot_2();  // 16-bit types
const GatherEntry *gather_stride_2();
// 4-byte elements, stride 2 or 4 (n <= 2^32): contiguous 256-bit span loads
// and a lane select; nullptr for other strides.
const GatherEntry *gather_span_4(int64_t stride);

// Bulk-copy (cp.async.bulk) staging variant of the streaming kernels: each
// CTA moves kTmaStages tiles of kTmaTile bytes per input through shared memory.
constexpr int kTmaTile = 8192;
constexpr int kTmaStages = 2;
constexpr int kTmaBlock = 128;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded mbarrier waits give up after 1 s

struct TmaArgs {
    const void *in0;
    const void *in1;
    void *out;
    int64_t n;
    int64_t head;     // elements [0, head) one by one (reach 16-byte alignment)
    int64_t ntiles;   // whole tiles after the head
    int64_t rem0;     // elements [rem0, n) one by one
    float alpha;
    uint64_t wait_limit_ns;
    int32_t shift0;   // realigning kernel: in0 + head*E lies shift0 bytes past a 16-byte boundary
    int32_t shift1;   // the same for in1 (the output is 16-byte aligned at element head)
};
using TmaLaunchFn = cudaError_t (*)(const TmaArgs &, int grid, cudaStream_t);
struct TmaEntry {
    const void *kernel;
    TmaLaunchFn launch;
    int smem_bytes;
};
// nullptr where no bulk-copy kernel exists for (op, dtype).
const TmaEntry *tma_entry(int op, int dtype);
// Realigning bulk-copy kernel: inputs at any element offset relative to the
// output.  Each input tile is copied as the 16-byte aligned span around it and
// read back at its offset in shared memory.  nullptr where none exists.
const TmaEntry *tma_realign_entry(int op, int dtype);
// One CTA that arms an mbarrier no copy will complete and must give up after
// limit_ns, recording error code 99 (checks the bounded-wait path).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s);
// Device error word written by bounded waits: read and cleared in one atomic
// exchange on the device, ordered on stream s.
cudaError_t read_and_clear_device_error(cudaStream_t s, int32_t *code);

}  // namespace ew
