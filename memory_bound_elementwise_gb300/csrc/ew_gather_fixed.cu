// ew_gather_fixed.cu -- instantiations of the fixed-stride tiled gather for
// strides below 32 that are not powers of two (both element sizes), in a
// translation unit of their own so that the build compiles them in parallel
// with the rest; ew_gather_fixed_wide.cu holds the strides from 33.
#include "ew_kernels.cuh"

namespace ew {

namespace {
#define EW_FIXED_STRIDES(X)                                                                        \
    X(3) X(5) X(6) X(7) X(9) X(10) X(11) X(12) X(13) X(14) X(15) X(17) X(18) X(19) X(20) X(21) \
    X(22) X(23) X(24) X(25) X(26) X(27) X(28) X(29) X(30) X(31)
#define EW_ENTRY4(S) tiled_fixed_entry<4, S, false>(),
#define EW_ENTRY2(S) tiled_fixed_entry<2, S, false>(),
#define EW_SHIFTED4(S) tiled_fixed_entry<4, S, true>(),
#define EW_SHIFTED2(S) tiled_fixed_entry<2, S, true>(),
#define EW_STRIDE(S) S,
const GatherEntry kFixed4[] = {EW_FIXED_STRIDES(EW_ENTRY4)};
const GatherEntry kFixed2[] = {EW_FIXED_STRIDES(EW_ENTRY2)};
const GatherEntry kShifted4[] = {EW_FIXED_STRIDES(EW_SHIFTED4)};  // input past a 16-byte boundary
const GatherEntry kShifted2[] = {EW_FIXED_STRIDES(EW_SHIFTED2)};
constexpr uint64_t kFixedStrides[] = {EW_FIXED_STRIDES(EW_STRIDE)};
// 2-byte elements at s = 2, 4 and 8 on an input past a 16-byte boundary
// (aligned ones take the power-of-two kernel).  Measured on GB300 at 2^26
// against the general kernel: bf16 +5.2%, +6.8% and +4.3%; at s = 16 and 32,
// and for fp32 at every power of two, -1.6% to +0.8%, so those keep it.
const GatherEntry kPow2Shifted2[] = {tiled_fixed_entry<2, 2, true>(), tiled_fixed_entry<2, 4, true>(),
                                     tiled_fixed_entry<2, 8, true>()};
#undef EW_ENTRY4
#undef EW_ENTRY2
#undef EW_SHIFTED4
#undef EW_SHIFTED2
#undef EW_STRIDE
#undef EW_FIXED_STRIDES
}  // namespace

// Every stride from 3 to 63 that is not a power of two; shifted, also
// 2-byte elements at s = 2, 4 and 8.
const GatherEntry *gather_tiled_fixed(int e, uint64_t stride, bool shifted) {
    if (stride > 32) return gather_tiled_fixed_wide(e, stride, shifted);
    if (shifted && e == 2 && (stride == 2 || stride == 4 || stride == 8))
        return &kPow2Shifted2[stride == 2 ? 0 : stride == 4 ? 1 : 2];
    for (size_t k = 0; k < sizeof(kFixedStrides) / sizeof(kFixedStrides[0]); ++k)
        if (kFixedStrides[k] == stride)
            return shifted ? (e == 4 ? &kShifted4[k] : &kShifted2[k]) : (e == 4 ? &kFixed4[k] : &kFixed2[k]);
    return nullptr;
}

}  // namespace ew
