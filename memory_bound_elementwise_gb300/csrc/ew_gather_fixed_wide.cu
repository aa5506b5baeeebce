// ew_gather_fixed_wide.cu -- instantiations of the fixed-stride tiled gather
// for the strides from 33 to 63 (both element sizes).
#include "ew_kernels.cuh"

namespace ew {

namespace {
#define EW_FIXED_STRIDES(X)                                                                        \
    X(33) X(34) X(35) X(36) X(37) X(38) X(39) X(40) X(41) X(42) X(43) X(44) X(45) X(46) X(47)  \
    X(48) X(49) X(50) X(51) X(52) X(53) X(54) X(55) X(56) X(57) X(58) X(59) X(60) X(61) X(62)  \
    X(63)
#define EW_ENTRY4(S) tiled_fixed_entry<4, S, false>(),
#define EW_ENTRY2(S) tiled_fixed_entry<2, S, false>(),
#define EW_SHIFTED4(S) tiled_fixed_entry<4, S, true>(),
#define EW_SHIFTED2(S) tiled_fixed_entry<2, S, true>(),
const GatherEntry kFixed4[] = {EW_FIXED_STRIDES(EW_ENTRY4)};
const GatherEntry kFixed2[] = {EW_FIXED_STRIDES(EW_ENTRY2)};
const GatherEntry kShifted4[] = {EW_FIXED_STRIDES(EW_SHIFTED4)};  // input past a 16-byte boundary
const GatherEntry kShifted2[] = {EW_FIXED_STRIDES(EW_SHIFTED2)};
#undef EW_ENTRY4
#undef EW_ENTRY2
#undef EW_SHIFTED4
#undef EW_SHIFTED2
#undef EW_FIXED_STRIDES
}  // namespace

const GatherEntry *gather_tiled_fixed_wide(int e, uint64_t stride, bool shifted) {
    if (stride < 33 || stride > 63) return nullptr;
    const size_t k = stride - 33;
    return shifted ? (e == 4 ? &kShifted4[k] : &kShifted2[k]) : (e == 4 ? &kFixed4[k] : &kFixed2[k]);
}

}  // namespace ew
