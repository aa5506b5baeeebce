// ew_kernels_bf16.cu -- bfloat16 instantiations of the streaming kernels
// (copy of 2-byte elements is shared with binary16).
#include "ew_kernels.cuh"

namespace ew {

namespace {
template <class Op>
constexpr StreamEntry eb(int vi) {
    return vi == 0 ? stream_entry<Op, 32>() : vi == 1 ? stream_entry<Op, 16>()
         : vi == 2 ? stream_entry<Op, 8>() : vi == 3 ? stream_entry<Op, 4>()
         : stream_entry<Op, 2>();
}

const StreamEntry kTable[OP_COUNT][5] = {
    {eb<OpAddBF16>(0), eb<OpAddBF16>(1), eb<OpAddBF16>(2), eb<OpAddBF16>(3), eb<OpAddBF16>(4)},
    {eb<OpSaxpyBF16>(0), eb<OpSaxpyBF16>(1), eb<OpSaxpyBF16>(2), eb<OpSaxpyBF16>(3), eb<OpSaxpyBF16>(4)},
    {eb<OpReluBF16>(0), eb<OpReluBF16>(1), eb<OpReluBF16>(2), eb<OpReluBF16>(3), eb<OpReluBF16>(4)},
    {kNoEntry, kNoEntry, kNoEntry, kNoEntry, kNoEntry},
    {eb<OpAddReluBF16>(0), eb<OpAddReluBF16>(1), eb<OpAddReluBF16>(2), eb<OpAddReluBF16>(3), eb<OpAddReluBF16>(4)},
    {kNoEntry, kNoEntry, kNoEntry, kNoEntry, kNoEntry},
    {eb<OpSaxpyReluBF16>(0), eb<OpSaxpyReluBF16>(1), eb<OpSaxpyReluBF16>(2), eb<OpSaxpyReluBF16>(3),
     eb<OpSaxpyReluBF16>(4)},
};
}  // namespace

const StreamEntry *stream_table_bf16() { return &kTable[0][0]; }

}  // namespace ew
