// ew_tma.cu -- bulk-copy staging variant of the streaming kernels, and the
// device error word that bounded waits report through.
//
// Each CTA owns kTmaStages consecutive tiles of kTmaTile bytes per input.
// Thread 0 arms one mbarrier per tile and issues every tile's global->shared
// bulk copy (cp.async.bulk ... mbarrier::complete_tx) up front; then, tile by
// tile, the CTA waits for the bytes, applies the operator in shared memory
// (result over the first input's buffer), makes the writes visible to the
// async proxy and thread 0 bulk-stores the tile (cp.async.bulk.global.shared).
// Latency is hidden across CTAs: many such CTAs are resident per SM and the
// block scheduler hands out the next tiles as CTAs finish.  No multicast, no
// clusters.  Elements before the first 16-byte aligned address and after the
// last whole tile are done one per thread by extra blocks after the tile
// blocks.
//
// Every mbarrier wait is bounded (%globaltimer): when it gives up the CTA
// records an error code, lets copies already in flight land (again bounded),
// drains its bulk stores and returns; the host reads the code with
// ew_device_error.
#include <atomic>
#include <mutex>
#include <type_traits>

#include "ew_internal.h"
#include "ew_kernels.cuh"

namespace ew {

__device__ int32_t g_device_error = 0;
// What the last read-and-clear took out of g_device_error (copied to the host).
__device__ int32_t g_device_error_taken = 0;

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(phase) : "memory");
    return done != 0;
}
// true when the phase completed, false when limit_ns passed first
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t phase, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, phase)) {
        if ((++spins & 255u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(smem_addr(src_smem)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_store_drain() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_to_async_proxy() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void record_error(int32_t code) { atomicCAS(&g_device_error, 0, code); }

// Blocks after the tile blocks take the elements outside the tiles, head
// [0, head) then remainder [rem0, n), one per thread.  Returns true in those
// blocks.
template <class Op>
__device__ __forceinline__ bool scalar_block(const Op &op, const TmaArgs &a, const char *in0, const char *in1,
                                             char *out) {
    const int64_t tile_blocks = (a.ntiles + kTmaStages - 1) / kTmaStages;
    if (static_cast<int64_t>(blockIdx.x) < tile_blocks) return false;
    const int64_t k = (static_cast<int64_t>(blockIdx.x) - tile_blocks) * kTmaBlock + threadIdx.x;
    const int64_t i = k < a.head ? k : a.rem0 + (k - a.head);
    if (i < a.n) apply_one(op, in0, in1, out, i * Op::kElem);
    return true;
}

template <class Op> struct IsCopy : std::false_type {};
template <int E> struct IsCopy<OpCopy<E>> : std::true_type {};

template <class Op>
__global__ void __launch_bounds__(kTmaBlock) tma_kernel(const TmaArgs a) {
    enter_grid();
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_failed;
    constexpr int NIN = Op::kIn, E = Op::kElem, T = kTmaTile, S = kTmaStages;
    unsigned char *buf0 = smem;
    unsigned char *buf1 = smem + S * T;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NIN * S * T);
    const Op op = make_op<Op>(a.alpha);
    const char *in0 = static_cast<const char *>(a.in0);
    const char *in1 = static_cast<const char *>(a.in1);
    char *out = static_cast<char *>(a.out);

    if (scalar_block(op, a, in0, in1, out)) return;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * S;
    const int cnt = static_cast<int>(a.ntiles - t0 < S ? a.ntiles - t0 : S);
    const char *g0 = in0 + a.head * E;
    const char *g1 = (NIN == 2) ? in1 + a.head * E : nullptr;
    char *go = out + a.head * E;

    if (threadIdx.x == 0) {
        s_failed = 0;
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int s = 0; s < cnt; ++s) {
            mbar_arrive_expect_tx(&full[s], NIN * T);
            bulk_load(buf0 + s * T, g0 + (t0 + s) * T, T, &full[s]);
            if constexpr (NIN == 2) bulk_load(buf1 + s * T, g1 + (t0 + s) * T, T, &full[s]);
        }
    }
    __syncthreads();
    int s = 0;
    for (; s < cnt; ++s) {
        if (threadIdx.x == 0 && !mbar_wait_bounded(&full[s], 0, a.wait_limit_ns)) {
            s_failed = 1;
            record_error(1);
        }
        __syncthreads();
        if (s_failed) break;
        if constexpr (!IsCopy<Op>::value) {
            uint4 *x4 = reinterpret_cast<uint4 *>(buf0 + s * T);
            const uint4 *y4 = reinterpret_cast<const uint4 *>(buf1 + s * T);
#pragma unroll
            for (int i = threadIdx.x; i < T / 16; i += kTmaBlock) {
                uint4 x = x4[i];
                const uint4 y = (NIN == 2) ? y4[i] : x;
                x.x = op.word(x.x, y.x);
                x.y = op.word(x.y, y.y);
                x.z = op.word(x.z, y.z);
                x.w = op.word(x.w, y.w);
                x4[i] = x;
            }
            fence_to_async_proxy();
            __syncthreads();
        }
        if (threadIdx.x == 0) bulk_store(go + (t0 + s) * T, buf0 + s * T, T);
    }
    if (threadIdx.x == 0) {
        bulk_store_drain();
        // After a wait gave up, let the loads still in flight land before the
        // CTA exits.  Only if this second wait expires too (both limits, 2 s in
        // all, with the memory system not delivering) does the CTA leave with
        // loads possibly still writing into its shared memory; the call's
        // outputs are then undefined, and code 1 in the error word says so.
        if (s_failed)
            for (int r = s; r < cnt; ++r) (void)mbar_wait_bounded(&full[r], 0, a.wait_limit_ns);
    }
}

// 16 bytes of a staged input that start `shift` bytes (even, < 16) past the
// i-th 16-byte chunk of its shared-memory buffer.  Two aligned 16-byte shared
// loads; a select of words by shift / 4; for shift = 2 mod 4, each output word
// joins the upper half of one word and the lower half of the next (prmt).
__device__ __forceinline__ uint4 load_shifted(const uint4 *buf, int i, int shift) {
    const uint4 lo = buf[i];
    const uint4 hi = shift != 0 ? buf[i + 1] : lo;
    const bool by8 = (shift & 8) != 0, by4 = (shift & 4) != 0;
    const uint32_t b0 = by8 ? lo.z : lo.x, b1 = by8 ? lo.w : lo.y, b2 = by8 ? hi.x : lo.z;
    const uint32_t b3 = by8 ? hi.y : lo.w, b4 = by8 ? hi.z : hi.x, b5 = by8 ? hi.w : hi.y;
    const uint32_t c0 = by4 ? b1 : b0, c1 = by4 ? b2 : b1, c2 = by4 ? b3 : b2;
    const uint32_t c3 = by4 ? b4 : b3, c4 = by4 ? b5 : b4;
    const uint32_t sel = (shift & 2) != 0 ? 0x5432u : 0x3210u;
    return make_uint4(__byte_perm(c0, c1, sel), __byte_perm(c1, c2, sel), __byte_perm(c2, c3, sel),
                      __byte_perm(c3, c4, sel));
}

// Bulk-copy kernel for inputs whose offsets differ from the output's modulo
// 16 bytes (where the aligned kernel cannot run).  The output tiles are
// 16-byte aligned.  For each input, the 16-byte aligned span around its tile
// (tile + 16 bytes when shift != 0) is bulk-copied to shared memory and read
// back at the input's shift.  The host keeps at least 16 bytes of elements
// outside the tiles at both ends, so each span lies inside its input array.
// Results go to a separate staging buffer per stage, bulk-stored as in
// tma_kernel.
template <class Op>
__global__ void __launch_bounds__(kTmaBlock) tma_realign_kernel(const TmaArgs a) {
    enter_grid();
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_failed;
    constexpr int NIN = Op::kIn, E = Op::kElem, T = kTmaTile, S = kTmaStages;
    constexpr int TI = T + 16;                // staged input span
    constexpr int kStage = NIN * TI + T;      // per stage: inputs, then the output tile
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * kStage);
    const Op op = make_op<Op>(a.alpha);
    const char *in0 = static_cast<const char *>(a.in0);
    const char *in1 = static_cast<const char *>(a.in1);
    char *out = static_cast<char *>(a.out);

    if (scalar_block(op, a, in0, in1, out)) return;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * S;
    const int cnt = static_cast<int>(a.ntiles - t0 < S ? a.ntiles - t0 : S);
    const int sh0 = a.shift0, sh1 = (NIN == 2) ? a.shift1 : 0;
    const char *g0 = in0 + a.head * E - sh0;  // 16-byte aligned
    const char *g1 = (NIN == 2) ? in1 + a.head * E - sh1 : nullptr;
    char *go = out + a.head * E;
    const uint32_t bytes0 = sh0 != 0 ? TI : T, bytes1 = sh1 != 0 ? TI : T;

    if (threadIdx.x == 0) {
        s_failed = 0;
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int s = 0; s < cnt; ++s) {
            unsigned char *st = smem + s * kStage;
            mbar_arrive_expect_tx(&full[s], bytes0 + (NIN == 2 ? bytes1 : 0u));
            bulk_load(st, g0 + (t0 + s) * T, bytes0, &full[s]);
            if constexpr (NIN == 2) bulk_load(st + TI, g1 + (t0 + s) * T, bytes1, &full[s]);
        }
    }
    __syncthreads();
    int s = 0;
    for (; s < cnt; ++s) {
        if (threadIdx.x == 0 && !mbar_wait_bounded(&full[s], 0, a.wait_limit_ns)) {
            s_failed = 1;
            record_error(1);
        }
        __syncthreads();
        if (s_failed) break;
        unsigned char *st = smem + s * kStage;
        const uint4 *x4 = reinterpret_cast<const uint4 *>(st);
        const uint4 *y4 = reinterpret_cast<const uint4 *>(st + TI);
        uint4 *o4 = reinterpret_cast<uint4 *>(st + NIN * TI);
#pragma unroll 4
        for (int i = threadIdx.x; i < T / 16; i += kTmaBlock) {
            const uint4 x = load_shifted(x4, i, sh0);
            const uint4 y = (NIN == 2) ? load_shifted(y4, i, sh1) : x;
            o4[i] = make_uint4(op.word(x.x, y.x), op.word(x.y, y.y), op.word(x.z, y.z), op.word(x.w, y.w));
        }
        fence_to_async_proxy();
        __syncthreads();
        if (threadIdx.x == 0) bulk_store(go + (t0 + s) * T, o4, T);
    }
    if (threadIdx.x == 0) {
        bulk_store_drain();
        // as in tma_kernel: loads may still be in flight at exit only after
        // both bounded waits expired, and code 1 then marks the outputs undefined
        if (s_failed)
            for (int r = s; r < cnt; ++r) (void)mbar_wait_bounded(&full[r], 0, a.wait_limit_ns);
    }
}

template <class Op>
constexpr int realign_smem_bytes() {
    return kTmaStages * (Op::kIn * (kTmaTile + 16) + kTmaTile) + kTmaStages * 8;
}

template <class Op>
cudaError_t launch_tma_realign(const TmaArgs &a, int grid, cudaStream_t s) {
    constexpr int smem = realign_smem_bytes<Op>();
    // above the 48 KiB default for two-input operators: opt in once per device
    static std::atomic<uint64_t> opted_in{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if ((opted_in.load(std::memory_order_acquire) & bit) == 0 || bit == 0) {
        e = cudaFuncSetAttribute(&tma_realign_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        opted_in.fetch_or(bit, std::memory_order_release);
    }
    return launch_kernel(&tma_realign_kernel<Op>, grid, kTmaBlock, smem, s, a);
}

template <class Op>
constexpr TmaEntry tma_realign_entry_of() {
    return TmaEntry{reinterpret_cast<const void *>(&tma_realign_kernel<Op>), &launch_tma_realign<Op>,
                    realign_smem_bytes<Op>()};
}

const TmaEntry kTmaRealign[OP_COUNT][DT_COUNT] = {
    {tma_realign_entry_of<OpAddF32>(), tma_realign_entry_of<OpAddF16>(), tma_realign_entry_of<OpAddBF16>()},
    {tma_realign_entry_of<OpSaxpyF32>(), tma_realign_entry_of<OpSaxpyF16>(),
     tma_realign_entry_of<OpSaxpyBF16>()},
    {tma_realign_entry_of<OpReluF32>(), tma_realign_entry_of<OpReluF16>(), tma_realign_entry_of<OpReluBF16>()},
    {tma_realign_entry_of<OpCopy<4>>(), tma_realign_entry_of<OpCopy<2>>(), tma_realign_entry_of<OpCopy<2>>()},
    {tma_realign_entry_of<OpAddReluF32>(), tma_realign_entry_of<OpAddReluF16>(),
     tma_realign_entry_of<OpAddReluBF16>()},
    {tma_realign_entry_of<OpSelectEvenOddI32>(), TmaEntry{nullptr, nullptr, 0}, TmaEntry{nullptr, nullptr, 0}},
    {tma_realign_entry_of<OpSaxpyReluF32>(), tma_realign_entry_of<OpSaxpyReluF16>(),
     tma_realign_entry_of<OpSaxpyReluBF16>()},
};

template <class Op>
cudaError_t launch_tma(const TmaArgs &a, int grid, cudaStream_t s) {
    constexpr int smem = Op::kIn * kTmaStages * kTmaTile + kTmaStages * 8;
    return launch_kernel(&tma_kernel<Op>, grid, kTmaBlock, smem, s, a);
}

template <class Op>
constexpr TmaEntry tma_entry_of() {
    return TmaEntry{reinterpret_cast<const void *>(&tma_kernel<Op>), &launch_tma<Op>,
                    Op::kIn * kTmaStages * kTmaTile + kTmaStages * 8};
}

const TmaEntry kTma[OP_COUNT][DT_COUNT] = {
    {tma_entry_of<OpAddF32>(), tma_entry_of<OpAddF16>(), tma_entry_of<OpAddBF16>()},
    {tma_entry_of<OpSaxpyF32>(), tma_entry_of<OpSaxpyF16>(), tma_entry_of<OpSaxpyBF16>()},
    {tma_entry_of<OpReluF32>(), tma_entry_of<OpReluF16>(), tma_entry_of<OpReluBF16>()},
    {tma_entry_of<OpCopy<4>>(), tma_entry_of<OpCopy<2>>(), tma_entry_of<OpCopy<2>>()},
    {tma_entry_of<OpAddReluF32>(), tma_entry_of<OpAddReluF16>(), tma_entry_of<OpAddReluBF16>()},
    {tma_entry_of<OpSelectEvenOddI32>(), TmaEntry{nullptr, nullptr, 0}, TmaEntry{nullptr, nullptr, 0}},
    {tma_entry_of<OpSaxpyReluF32>(), tma_entry_of<OpSaxpyReluF16>(), tma_entry_of<OpSaxpyReluBF16>()},
};

// Arms an mbarrier for 16 bytes that no copy will deliver: the bounded wait
// must give up, record code 99 and return.  Nothing is in flight.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    enter_grid();
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        mbar_arrive_expect_tx(&bar, 16);
        if (!mbar_wait_bounded(&bar, 0, limit_ns)) record_error(99);
    }
}

// Moves the error word out (leaving 0) in one atomic exchange, so a code that
// a kernel on another stream records meanwhile is kept for the next read.
__global__ void take_device_error_kernel() {
    enter_grid();
    g_device_error_taken = atomicExch(&g_device_error, 0);
}

std::mutex g_take_mu;  // one reader of g_device_error_taken at a time

}  // namespace

const TmaEntry *tma_entry(int op, int dtype) {
    if (op < 0 || op >= OP_COUNT || dtype < 0 || dtype >= DT_COUNT) return nullptr;
    const TmaEntry *e = &kTma[op][dtype];
    return e->launch != nullptr ? e : nullptr;
}

const TmaEntry *tma_realign_entry(int op, int dtype) {
    if (op < 0 || op >= OP_COUNT || dtype < 0 || dtype >= DT_COUNT) return nullptr;
    const TmaEntry *e = &kTmaRealign[op][dtype];
    return e->launch != nullptr ? e : nullptr;
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
    return launch_kernel(&wait_selftest_kernel, 1, 32, 0, s, limit_ns);
}

cudaError_t read_and_clear_device_error(cudaStream_t s, int32_t *code) {
    std::lock_guard<std::mutex> lk(g_take_mu);
    int32_t v = 0;
    cudaError_t e = launch_kernel(&take_device_error_kernel, 1, 1, 0, s);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbolAsync(&v, g_device_error_taken, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    *code = v;
    return e;
}

}  // namespace ew
