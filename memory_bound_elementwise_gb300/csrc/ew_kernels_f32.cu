// ew_kernels_f32.cu -- 4-byte instantiations of the streaming kernels
// (binary32 operators, the int32 even/odd select, 4-byte copy) and the 4-byte
// strided gather.
#include "ew_kernels.cuh"

namespace ew {

namespace {
template <class Op>
constexpr StreamEntry e32(int vi) {
    return vi == 0 ? stream_entry<Op, 32>() : vi == 1 ? stream_entry<Op, 16>()
         : vi == 2 ? stream_entry<Op, 8>() : vi == 3 ? stream_entry<Op, 4>() : kNoEntry;
}
const StreamEntry kTable[OP_COUNT][5] = {
    {e32<OpAddF32>(0), e32<OpAddF32>(1), e32<OpAddF32>(2), e32<OpAddF32>(3), kNoEntry},
    {e32<OpSaxpyF32>(0), e32<OpSaxpyF32>(1), e32<OpSaxpyF32>(2), e32<OpSaxpyF32>(3), kNoEntry},
    {e32<OpReluF32>(0), e32<OpReluF32>(1), e32<OpReluF32>(2), e32<OpReluF32>(3), kNoEntry},
    {e32<OpCopy<4>>(0), e32<OpCopy<4>>(1), e32<OpCopy<4>>(2), e32<OpCopy<4>>(3), kNoEntry},
    {e32<OpAddReluF32>(0), e32<OpAddReluF32>(1), e32<OpAddReluF32>(2), e32<OpAddReluF32>(3), kNoEntry},
    {e32<OpSelectEvenOddI32>(0), e32<OpSelectEvenOddI32>(1), e32<OpSelectEvenOddI32>(2),
     e32<OpSelectEvenOddI32>(3), kNoEntry},
    {e32<OpSaxpyReluF32>(0), e32<OpSaxpyReluF32>(1), e32<OpSaxpyReluF32>(2), e32<OpSaxpyReluF32>(3), kNoEntry},
};

constexpr int kGatherOneshotUnroll = 4;
constexpr int kGatherStrideUnroll = 8;
const GatherEntry kGatherOneshot{reinterpret_cast<const void *>(&gather_oneshot_kernel<4, kGatherOneshotUnroll>),
                                 &launch_gather_oneshot<4, kGatherOneshotUnroll>, kGatherOneshotUnroll};
const GatherEntry kGatherStride{reinterpret_cast<const void *>(&gather_stride_kernel<4, kGatherStrideUnroll>),
                                &launch_gather_stride<4, kGatherStrideUnroll>, kGatherStrideUnroll};
constexpr int kGatherLapsUnroll = 8;
const GatherEntry kGatherLaps{reinterpret_cast<const void *>(&gather_laps_kernel<4, kGatherLapsUnroll>),
                              &launch_gather_laps<4, kGatherLapsUnroll>, kGatherLapsUnroll};
constexpr int kGatherTiledUnroll = 2;  // 16-byte loads in flight per thread per batch
const GatherEntry kGatherTiled{reinterpret_cast<const void *>(&gather_tiled_kernel<4, kGatherTiledUnroll>),
                               &launch_gather_tiled<4, kGatherTiledUnroll>, kGatherTiledUnroll};
}  // namespace

const StreamEntry *stream_table_f32() { return &kTable[0][0]; }

constexpr int kGatherSpanUnroll = 2;
static const GatherEntry kGatherSpan2{reinterpret_cast<const void *>(&gather_span_kernel<2, kGatherSpanUnroll>),
                               &launch_gather_span<2, kGatherSpanUnroll>, kGatherSpanUnroll};
static const GatherEntry kGatherSpan4{reinterpret_cast<const void *>(&gather_span_kernel<4, kGatherSpanUnroll>),
                               &launch_gather_span<4, kGatherSpanUnroll>, kGatherSpanUnroll};

const GatherEntry *gather_span_4(int64_t stride) {
    return stride == 2 ? &kGatherSpan2 : stride == 4 ? &kGatherSpan4 : nullptr;
}
const GatherEntry *gather_oneshot_4() { return &kGatherOneshot; }
const GatherEntry *gather_laps_4() { return &kGatherLaps; }
const GatherEntry *gather_tiled_4() { return &kGatherTiled; }

static const GatherEntry kGatherTiledPow2[6] = {tiled_pow2_entry<4, 2>(), tiled_pow2_entry<4, 4>(),
                                                tiled_pow2_entry<4, 8>(), tiled_pow2_entry<4, 16>(),
                                                tiled_pow2_entry<4, 32>(), tiled_pow2_entry<4, 64>()};

const GatherEntry *gather_tiled_pow2_4(uint64_t stride) {
    switch (stride) {
        case 2: return &kGatherTiledPow2[0];
        case 4: return &kGatherTiledPow2[1];
        case 8: return &kGatherTiledPow2[2];
        case 16: return &kGatherTiledPow2[3];
        case 32: return &kGatherTiledPow2[4];
        case 64: return &kGatherTiledPow2[5];
        default: return nullptr;
    }
}
const GatherEntry *gather_stride_4() { return &kGatherStride; }

}  // namespace ew
