// ew_kernels_f16.cu -- binary16 instantiations of the streaming kernels, the
// 2-byte copy (shared by binary16 and bfloat16) and the 2-byte strided gather.
#include "ew_kernels.cuh"

namespace ew {

namespace {
template <class Op>
constexpr StreamEntry e16(int vi) {
    return vi == 0 ? stream_entry<Op, 32>() : vi == 1 ? stream_entry<Op, 16>()
         : vi == 2 ? stream_entry<Op, 8>() : vi == 3 ? stream_entry<Op, 4>()
         : stream_entry<Op, 2>();
}

const StreamEntry kTable[OP_COUNT][5] = {
    {e16<OpAddF16>(0), e16<OpAddF16>(1), e16<OpAddF16>(2), e16<OpAddF16>(3), e16<OpAddF16>(4)},
    {e16<OpSaxpyF16>(0), e16<OpSaxpyF16>(1), e16<OpSaxpyF16>(2), e16<OpSaxpyF16>(3), e16<OpSaxpyF16>(4)},
    {e16<OpReluF16>(0), e16<OpReluF16>(1), e16<OpReluF16>(2), e16<OpReluF16>(3), e16<OpReluF16>(4)},
    {e16<OpCopy<2>>(0), e16<OpCopy<2>>(1), e16<OpCopy<2>>(2), e16<OpCopy<2>>(3), e16<OpCopy<2>>(4)},
    {e16<OpAddReluF16>(0), e16<OpAddReluF16>(1), e16<OpAddReluF16>(2), e16<OpAddReluF16>(3), e16<OpAddReluF16>(4)},
    {kNoEntry, kNoEntry, kNoEntry, kNoEntry, kNoEntry},
    {e16<OpSaxpyReluF16>(0), e16<OpSaxpyReluF16>(1), e16<OpSaxpyReluF16>(2), e16<OpSaxpyReluF16>(3),
     e16<OpSaxpyReluF16>(4)},
};

constexpr int kGatherOneshotUnroll = 4;
constexpr int kGatherStrideUnroll = 8;
const GatherEntry kGatherOneshot{reinterpret_cast<const void *>(&gather_oneshot_kernel<2, kGatherOneshotUnroll>),
                                 &launch_gather_oneshot<2, kGatherOneshotUnroll>, kGatherOneshotUnroll};
const GatherEntry kGatherStride{reinterpret_cast<const void *>(&gather_stride_kernel<2, kGatherStrideUnroll>),
                                &launch_gather_stride<2, kGatherStrideUnroll>, kGatherStrideUnroll};
constexpr int kGatherLapsUnroll = 8;
const GatherEntry kGatherLaps{reinterpret_cast<const void *>(&gather_laps_kernel<2, kGatherLapsUnroll>),
                              &launch_gather_laps<2, kGatherLapsUnroll>, kGatherLapsUnroll};
constexpr int kGatherTiledUnroll = 2;  // 16-byte loads in flight per thread per batch
const GatherEntry kGatherTiled{reinterpret_cast<const void *>(&gather_tiled_kernel<2, kGatherTiledUnroll>),
                               &launch_gather_tiled<2, kGatherTiledUnroll>, kGatherTiledUnroll};
}  // namespace

const StreamEntry *stream_table_f16() { return &kTable[0][0]; }

const GatherEntry *gather_oneshot_2() { return &kGatherOneshot; }
const GatherEntry *gather_laps_2() { return &kGatherLaps; }
const GatherEntry *gather_tiled_2() { return &kGatherTiled; }

static const GatherEntry kGatherTiledPow2[6] = {tiled_pow2_entry<2, 2>(), tiled_pow2_entry<2, 4>(),
                                                tiled_pow2_entry<2, 8>(), tiled_pow2_entry<2, 16>(),
                                                tiled_pow2_entry<2, 32>(), tiled_pow2_entry<2, 64>()};

const GatherEntry *gather_tiled_pow2_2(uint64_t stride) {
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
const GatherEntry *gather_stride_2() { return &kGatherStride; }

}  // namespace ew
