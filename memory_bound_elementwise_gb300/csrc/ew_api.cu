// ew_api.cu -- the C ABI declared in include/ew.h: argument validation,
// alignment planning, launch geometry and dispatch to the kernel tables.
//
// Validation happens entirely on the host, before any CUDA runtime call, so
// argument errors never reach the GPU.
//
// Launch geometry.  The body is cut into chunks of kBlock threads x U vectors
// ("逐元素操作算子" §二: the launch is sized from N with a ceil-div, and a
// grid-stride loop decouples the grid from N).  One-shot schedule (default):
// one block per chunk, so the block scheduler keeps every SM busy until the
// last chunk (CUDA-MODE lecture notes §4.2: a partial last wave idles SMs; here
// the waves are many and short).  Persistent schedule: SMs x resident blocks
// per SM from the occupancy API (CUDA-MODE lecture notes §4.4), each block
// striding over the chunks.
#include <algorithm>
#include <array>
#include <atomic>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include <cuda_runtime.h>

#include "ew.h"
#include "ew_internal.h"

using namespace ew;

namespace {

std::atomic<int> g_path{EW_PATH_AUTO};
std::atomic<int> g_schedule{EW_SCHED_AUTO};
std::atomic<int> g_pointer_check{-1};  // -1: not yet read from the environment
std::atomic<int> g_programmatic{1};

thread_local int t_last_cuda_error = 0;
thread_local ew_launch_record t_last{};

int elem_size(ew_dtype dt) { return (dt == EW_F32 || dt == EW_I32) ? 4 : 2; }
bool dtype_ok(int dt) { return dt == EW_F32 || dt == EW_F16 || dt == EW_BF16 || dt == EW_I32; }
bool float_dtype(ew_dtype dt) { return dt == EW_F32 || dt == EW_F16 || dt == EW_BF16; }
// the kernel tables are per element size: int32 shares the 4-byte table
int table_dtype(ew_dtype dt) { return dt == EW_I32 ? DT_F32 : static_cast<int>(dt); }

ew_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return EW_ERR_CUDA;
}

// byte ranges [p, p+len) and [q, q+len) share a byte
bool overlaps(const void *p, const void *q, int64_t len) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + static_cast<uintptr_t>(len) && b < a + static_cast<uintptr_t>(len);
}

// ---------------------------------------------------------------- planning

// AUTO's access width for the vector body is 32 bytes (the widest the
// pointers share).  Measured on GB300 through this library in alternating
// blocks of 50 launches of one width (2^25 to 2^28 elements; add, SAXPY,
// ReLU, copy in fp32 and bf16), 16- and 32-byte accesses with 64 bytes in
// flight per thread per input tie within 0.6% in most cases; the 32-byte
// kernels are 0.2-0.6% ahead for the fp32 add and SAXPY from 2^26, the
// 16-byte ones 1.5-2% ahead for bf16 ReLU and copy at 2^26-2^27.  The 32-byte
// kernels issue half as many memory instructions and keep the three-operand
// fp32 operators ahead, so AUTO keeps them.
int path_cap_bytes(int path, int e) {
    switch (path) {
        case EW_PATH_SCALAR: return e;
        case EW_PATH_V128: return 16;
        default: return 32;  // AUTO, V256, TMA
    }
}

// Widest vector width (<= cap) at which all pointers sit at the same offset;
// the head brings that common offset to zero.
ew_plan make_plan(int path, int e, const uintptr_t *p, int np, int64_t n) {
    int vb = e;
    for (int w = path_cap_bytes(path, e); w > e; w >>= 1) {
        bool same = true;
        for (int k = 1; k < np; ++k) same = same && (p[k] % w == p[0] % w);
        if (same) { vb = w; break; }
    }
    ew_plan pl{};
    pl.vec_bytes = vb;
    int64_t head = (vb == e) ? 0 : static_cast<int64_t>((vb - p[0] % vb) % vb) / e;
    head = std::min<int64_t>(head, n);
    const int64_t per = vb / e;
    pl.head = head;
    pl.nvec = (n - head) / per;
    pl.tail = n - head - pl.nvec * per;
    pl.path = (vb == 32) ? EW_PATH_V256 : (vb == 16) ? EW_PATH_V128 : EW_PATH_SCALAR;
    return pl;
}

int selected_path() { return g_path.load(std::memory_order_relaxed); }
// schedule of the streaming kernels (lap order exists for the gather only)
int resolved_schedule() {
    const int s = g_schedule.load(std::memory_order_relaxed);
    return (s == EW_SCHED_AUTO || s == EW_SCHED_LAPS || s == EW_SCHED_TILED) ? EW_SCHED_ONESHOT : s;
}

// Bulk-copy split: 16-byte aligned head, whole tiles, then the remainder.
struct TmaPlan { int64_t head, ntiles, rem0; };

// Blocks of a bulk-copy launch: kTmaStages tiles per block, then one block per
// kTmaBlock elements outside the tiles (head and remainder, one per thread).
int64_t tma_grid(const TmaPlan &tp, int64_t n) {
    const int64_t scalar = tp.head + (n - tp.rem0);
    return (tp.ntiles + kTmaStages - 1) / kTmaStages + (scalar + kTmaBlock - 1) / kTmaBlock;
}

// The bulk-copy launches have no grid-stride loop: they need a grid of at most
// INT_MAX blocks (arrays below 2^31 x 16 KiB); beyond it the vector kernels run.
bool tma_grid_fits(int64_t n, int e) {
    return n / (kTmaTile / e) / kTmaStages < INT_MAX - 2 * kTmaTile;
}
TmaPlan make_tma_plan(const ew_plan &pl16, int e, int64_t n) {
    TmaPlan t{};
    t.head = pl16.head;
    const int64_t per_tile = kTmaTile / e;
    t.ntiles = (n - t.head) / per_tile;
    t.rem0 = t.head + t.ntiles * per_tile;
    return t;
}

// ---------------------------------------------------------------- devices

struct DevInfo { int sms = 0; int pageable_access = 0; };
std::mutex g_mu;
std::map<int, DevInfo> g_dev;
std::map<std::pair<int, const void *>, int> g_occ;

cudaError_t device_info(int *dev, int *sms, int *pageable_access = nullptr) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(*dev);
    if (it == g_dev.end()) {
        DevInfo d;
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&d.pageable_access, cudaDevAttrPageableMemoryAccess, *dev);
        if (e != cudaSuccess) return e;
        it = g_dev.emplace(*dev, d).first;
    }
    *sms = it->second.sms;
    if (pageable_access) *pageable_access = it->second.pageable_access;
    return cudaSuccess;
}

cudaError_t blocks_per_sm(int dev, const void *kernel, int block, int smem, int *out) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, kernel);
    auto it = g_occ.find(key);
    if (it == g_occ.end()) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, block, smem);
        if (e != cudaSuccess) return e;
        it = g_occ.emplace(key, std::max(b, 1)).first;
    }
    *out = it->second;
    return cudaSuccess;
}

bool pointer_check_enabled() {
    int v = g_pointer_check.load(std::memory_order_relaxed);
    if (v < 0) {
        const char *s = std::getenv("EW_CHECK_POINTERS");
        v = (s && s[0] == '1') ? 1 : 0;
        g_pointer_check.store(v, std::memory_order_relaxed);
    }
    return v == 1;
}

// Device memory, managed memory and page-locked host memory are reachable
// from kernels; plain pageable host memory only where the device reports
// pageable memory access (e.g. coherent CPU-GPU systems).
ew_status check_device_pointers(const void *const *p, int np) {
    int dev = 0, sms = 0, pageable = 0;
    cudaError_t e = device_info(&dev, &sms, &pageable);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int k = 0; k < np; ++k) {
        cudaPointerAttributes at{};
        e = cudaPointerGetAttributes(&at, p[k]);
        if (e != cudaSuccess) { cudaGetLastError(); return EW_ERR_NOT_DEVICE_POINTER; }
        const bool reachable = at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged ||
                               at.type == cudaMemoryTypeHost ||
                               (at.type == cudaMemoryTypeUnregistered && pageable == 1);
        if (!reachable) return EW_ERR_NOT_DEVICE_POINTER;
    }
    return EW_OK;
}

// True while s is being captured into a CUDA graph, or when that cannot be
// told.  AUTO then keeps the vector kernels rather than query pointers inside
// a capture.
bool stream_capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return st != cudaStreamCaptureStatusNone;
}

// True when every pointer is device memory.  AUTO sends bulk copies only
// there: host memory reached over the CPU-GPU link keeps the vector kernels.
bool all_device_memory(const void *const *p, int np) {
    for (int k = 0; k < np; ++k) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, p[k]) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (at.type != cudaMemoryTypeDevice) return false;
    }
    return true;
}

// Row padding, in 4-byte words, of the general tiled gather's tile.  Lane t
// of warp w stores element k of its 16-byte load, span element
// j = V*(32*w + t) + k (V elements per load), to row j mod s, column j / s.
// Rows are p elements (a multiple of 32 words) plus w_pad words apart, so the
// element lands in bank ((j mod s) * w_pad + word of j / s) mod 32.  Chosen
// once per (s, element size, p): the w_pad in [1, 32) with the fewest
// wavefronts (the most distinct words in one bank) summed over the stores of
// a whole span.  An input past a 16-byte boundary shifts j by the same few
// elements in every load, which moves no store into another bank count.
uint32_t tiled_pad_words(uint32_t s, int e, uint32_t p) {
    static std::mutex mu;
    static std::map<std::pair<int, uint32_t>, uint32_t> cache;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(e, s);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const uint32_t v = 16 / static_cast<uint32_t>(e), ew = static_cast<uint32_t>(e);
    const uint32_t nv = s * p / v;  // loads in a full span
    uint32_t best_w = 1;
    uint64_t best = ~uint64_t(0);
    for (uint32_t w_pad = 1; w_pad < 32; ++w_pad) {
        uint64_t total = 0;
        for (uint32_t w = 0; w * 32 < nv; ++w) {
            for (uint32_t k = 0; k < v; ++k) {
                uint32_t words[32], nw = 0, per_bank[32] = {}, worst = 0;
                for (uint32_t t = 0; t < 32 && 32 * w + t < nv; ++t) {
                    const uint32_t j = v * (32 * w + t) + k;
                    const uint32_t word = (j % s) * (2048 + w_pad) + (j / s) * ew / 4;
                    bool seen = false;
                    for (uint32_t q = 0; q < nw; ++q) seen = seen || words[q] == word;
                    if (!seen) {
                        words[nw++] = word;
                        worst = std::max(worst, ++per_bank[word % 32]);
                    }
                }
                total += worst;
            }
        }
        if (total < best) {
            best = total;
            best_w = w_pad;
        }
    }
    cache.emplace(key, best_w);
    return best_w;
}

// Row padding, in elements, of the fixed-stride tiled gather's tile: the pad
// in [0, 32) (even for 2-byte elements, so rows start on whole words) that
// minimises the most distinct words any bank receives when the lanes of a
// warp store element k of their 16-byte loads, over every warp of the block
// and every k.  Computed once per (element size, stride).
uint32_t fixed_pad_elems(int e, uint32_t s, uint32_t p, uint32_t threads) {
    static std::mutex mu;
    static std::map<std::pair<int, uint32_t>, uint32_t> cache;
    std::lock_guard<std::mutex> lk(mu);
    const auto key = std::make_pair(e, s);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const uint32_t v = 16 / static_cast<uint32_t>(e), step = e == 2 ? 2 : 1;
    uint32_t best_pad = 0, best = ~0u;
    for (uint32_t pad = 0; pad < 32; pad += step) {
        uint32_t worst = 0;
        for (uint32_t w = 0; 32 * w < threads; ++w) {  // a partial last warp too
            for (uint32_t k = 0; k < v; ++k) {
                uint32_t words[32], nw = 0, per_bank[32] = {};
                for (uint32_t t = 0; t < 32 && 32 * w + t < threads; ++t) {
                    const uint32_t j = v * (32 * w + t) + k;
                    const uint32_t word = ((j % s) * (p + pad) + j / s) * static_cast<uint32_t>(e) / 4;
                    bool seen = false;
                    for (uint32_t q = 0; q < nw; ++q) seen = seen || words[q] == word;
                    if (!seen) {
                        words[nw++] = word;
                        worst = std::max(worst, ++per_bank[word % 32]);
                    }
                }
            }
        }
        if (worst < best) {
            best = worst;
            best_pad = pad;
        }
    }
    cache.emplace(key, best_pad);
    return best_pad;
}

int clamp_grid(int64_t blocks) {
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(blocks, INT_MAX)));
}

// ---------------------------------------------------------------- dispatch

const StreamEntry *table_for(int tdt) {
    return tdt == DT_F32 ? stream_table_f32() : tdt == DT_F16 ? stream_table_f16() : stream_table_bf16();
}

ew_status run_tma(int op, ew_dtype dt, const void *in0, const void *in1, void *out, int64_t n,
                  float alpha, const ew_plan &pl16, cudaStream_t s) {
    const TmaEntry *ent = tma_entry(op, table_dtype(dt));
    const int e = elem_size(dt);
    const TmaPlan tp = make_tma_plan(pl16, e, n);
    TmaArgs a{in0, in1, out, n, tp.head, tp.ntiles, tp.rem0, alpha, kWaitLimitNs, 0, 0};
    const int grid = static_cast<int>(tma_grid(tp, n));
    cudaError_t ce = ent->launch(a, grid, s);
    if (ce != cudaSuccess) return cuda_fail(ce);
    t_last.launches = 1;
    t_last.path = EW_PATH_TMA;
    t_last.vec_bytes = 16;
    t_last.grid = grid;
    t_last.block = kTmaBlock;
    t_last.smem = ent->smem_bytes;
    t_last.schedule = EW_SCHED_ONESHOT;
    t_last.head = tp.head;
    t_last.nvec = tp.ntiles;
    t_last.tail = n - tp.rem0;
    return EW_OK;
}

// Realigning bulk-copy split, for pointers that disagree modulo 16 bytes:
// output tiles start 16-byte aligned, and each input is staged as the aligned
// span around its tile.  At least 16 bytes of elements stay outside the tiles
// at both ends, so the spans never leave the input arrays.
TmaPlan make_realign_plan(uintptr_t out, int e, int64_t n) {
    TmaPlan t{};
    t.head = static_cast<int64_t>((16 - out % 16) % 16) / e;
    if (t.head * e < 16) t.head += 16 / e;
    const int64_t per_tile = kTmaTile / e;
    const int64_t avail = n - t.head - 16 / e;
    t.ntiles = avail > 0 ? avail / per_tile : 0;
    if (t.ntiles == 0) t.head = std::min<int64_t>(t.head, n);
    t.rem0 = t.head + t.ntiles * per_tile;
    return t;
}

// Under EW_PATH_AUTO, 16-bit operands whose pointers differ in parity (2-byte
// accesses otherwise) take the realigning bulk-copy kernel from this size on.
constexpr int64_t kRealignAutoMinElems = int64_t(1) << 22;

bool auto_realign(int e, const ew_plan &pl, int64_t n) {
    return g_path.load(std::memory_order_relaxed) == EW_PATH_AUTO && e == 2 && pl.vec_bytes == 2 &&
           n >= kRealignAutoMinElems;
}

ew_status run_tma_realign(int op, ew_dtype dt, const void *in0, const void *in1, void *out, int64_t n,
                          float alpha, cudaStream_t s) {
    const TmaEntry *ent = tma_realign_entry(op, table_dtype(dt));
    const int e = elem_size(dt);
    const TmaPlan tp = make_realign_plan(reinterpret_cast<uintptr_t>(out), e, n);
    const int64_t head = tp.head, ntiles = tp.ntiles, rem0 = tp.rem0;
    const int32_t shift0 = static_cast<int32_t>((reinterpret_cast<uintptr_t>(in0) + head * e) % 16);
    const int32_t shift1 =
        in1 != nullptr ? static_cast<int32_t>((reinterpret_cast<uintptr_t>(in1) + head * e) % 16) : 0;
    TmaArgs a{in0, in1, out, n, head, ntiles, rem0, alpha, kWaitLimitNs, shift0, shift1};
    const int grid = static_cast<int>(tma_grid(tp, n));
    cudaError_t ce = ent->launch(a, grid, s);
    if (ce != cudaSuccess) return cuda_fail(ce);
    t_last.launches = 1;
    t_last.path = EW_PATH_TMA;
    t_last.vec_bytes = 16;
    t_last.grid = grid;
    t_last.block = kTmaBlock;
    t_last.smem = ent->smem_bytes;
    t_last.schedule = EW_SCHED_ONESHOT;
    t_last.head = head;
    t_last.nvec = ntiles;
    t_last.tail = n - rem0;
    return EW_OK;
}

// Common path of add / saxpy / relu / copy once arguments are valid.
ew_status run_stream(int op, ew_dtype dt, const void *in0, const void *in1, void *out,
                     int64_t n, float alpha, cudaStream_t s, bool skip_unchanged = false) {
    const int e = elem_size(dt);
    const void *ptrs[3] = {in0, out, in1};
    const int np = (in1 != nullptr) ? 3 : 2;
    uintptr_t up[3];
    for (int k = 0; k < np; ++k) up[k] = reinterpret_cast<uintptr_t>(ptrs[k]);
    const int path = selected_path();
    const ew_plan pl = make_plan(path, e, up, np, n);

    if (pointer_check_enabled()) {
        ew_status st = check_device_pointers(ptrs, np);
        if (st != EW_OK) return st;
    }
    int dev = 0, sms = 0;
    cudaError_t ce = device_info(&dev, &sms);
    if (ce != cudaSuccess) return cuda_fail(ce);

    if (path == EW_PATH_TMA && tma_entry(op, table_dtype(dt)) != nullptr && tma_grid_fits(n, e)) {
        if (pl.vec_bytes >= 16)
            return run_tma(op, dt, in0, in1, out, n, alpha, make_plan(EW_PATH_V128, e, up, np, n), s);
        return run_tma_realign(op, dt, in0, in1, out, n, alpha, s);
    }
    if (auto_realign(e, pl, n) && tma_realign_entry(op, table_dtype(dt)) != nullptr && tma_grid_fits(n, e) &&
        !stream_capturing(s) && all_device_memory(ptrs, np))
        return run_tma_realign(op, dt, in0, in1, out, n, alpha, s);

    StreamArgs a{in0, in1, out, n, pl.head, pl.nvec, pl.head + pl.nvec * (pl.vec_bytes / e), alpha,
                 skip_unchanged ? 1 : 0};

    // copy of 16-bit elements is one kernel for both 16-bit formats
    const int tdt = (op == OP_COPY && dt == EW_BF16) ? DT_F16 : table_dtype(dt);
    const StreamEntry &ent = table_for(tdt)[op * 5 + vec_index(pl.vec_bytes)];
    if (ent.launch == nullptr) return EW_ERR_INVALID_VALUE;

    const int64_t per_block = static_cast<int64_t>(kBlock) * ent.unroll;
    const int64_t nchunks = (pl.nvec + per_block - 1) / per_block;
    const int sched = resolved_schedule();
    int64_t blocks = nchunks;
    if (sched == EW_SCHED_PERSISTENT) {
        int occ = 1;
        ce = blocks_per_sm(dev, ent.kernel, kBlock, 0, &occ);
        if (ce != cudaSuccess) return cuda_fail(ce);
        blocks = std::min<int64_t>(nchunks, static_cast<int64_t>(sms) * occ);
    }
    const int grid = clamp_grid(blocks);

    ce = ent.launch(a, grid, s);
    if (ce != cudaSuccess) return cuda_fail(ce);
    t_last.launches = 1;
    t_last.path = pl.path;
    t_last.vec_bytes = pl.vec_bytes;
    t_last.grid = grid;
    t_last.block = kBlock;
    t_last.smem = 0;
    t_last.schedule = sched;
    t_last.head = pl.head;
    t_last.nvec = pl.nvec;
    t_last.tail = pl.tail;
    return EW_OK;
}

// Shared argument checks: dtype, n, null pointers, element alignment.
ew_status check_common(ew_dtype dt, int64_t n, const void *const *p, int np) {
    if (!dtype_ok(static_cast<int>(dt))) return EW_ERR_UNSUPPORTED_DTYPE;
    if (n < 0) return EW_ERR_INVALID_VALUE;
    if (n == 0) return EW_OK;
    for (int k = 0; k < np; ++k)
        if (p[k] == nullptr) return EW_ERR_NULL_POINTER;
    const uintptr_t e = static_cast<uintptr_t>(elem_size(dt));
    for (int k = 0; k < np; ++k)
        if (reinterpret_cast<uintptr_t>(p[k]) % e != 0) return EW_ERR_INVALID_VALUE;
    if (n > INT64_MAX / 8) return EW_ERR_INVALID_VALUE;
    return EW_OK;
}

// An output may equal an input exactly; any other shared byte is an error.
ew_status check_alias(const void *in, const void *out, int64_t bytes) {
    if (in == out) return EW_OK;
    return overlaps(in, out, bytes) ? EW_ERR_OVERLAP : EW_OK;
}

// ---------------------------------------------------------------- gather planning

// One gather launch: kernel, arguments, grid and what the launch record reports.
struct GatherLaunch {
    const GatherEntry *entry = nullptr;
    GatherArgs args{};
    int grid = 0, block = kBlock;
    int32_t path = EW_PATH_SCALAR, vec_bytes = 0, smem = 0, schedule = EW_SCHED_ONESHOT;
    int64_t head = 0, nvec = 0, tail = 0;
};

enum class GatherKind { SPAN, TILED, LAPS, ONESHOT, STRIDE };

constexpr uint64_t kOneshotMaxN = uint64_t(1) << 32;  // the 32-bit index kernels

// AUTO's crossover from lap order to the tiled kernels.  Lap order issues one
// load per output: as s grows each fp32 lane's load needs more of its own
// 32-byte sector (from s = 8 one per lane; L2-to-SM traffic bounds it), and
// 16-bit lanes move 2 bytes per load.  The tiled kernels read 16 bytes per
// load at any s.  Measured on GB300 at 2^26 elements they win from s = 5 for
// both element sizes (fp32 at s = 5, 6, 7: 6396, 6399, 6480 GB/s against
// 6101, 5941, 5463 in lap order), and lap order stays 2-3% ahead below that.
// For 2-byte elements the tiled kernels win from s = 2: at s = 2, 3 and 4
// the kernels specialised for the stride on a 16-byte aligned input (bf16:
// 5974, 5866, 5996 GB/s against 5358, 4998, 5239 in lap order), and on an
// input past a 16-byte boundary the fixed-stride kernel's shifted instances
// (5948, 5906, 6045 against 5375, 4973, 5235).
bool auto_tiled(int e, uint64_t s_mod) { return s_mod >= (e == 2 ? 2u : 5u); }

GatherArgs gather_args(const void *in, void *out, uint64_t n, uint64_t s_mod) {
    GatherArgs a{};
    a.in = in;
    a.out = out;
    a.n = n;
    a.s_mod = s_mod;
    return a;
}

// The lap geometry shared by the lap-ordered and tiled kernels:
// n = lap_q * s + lap_m, and division by s through floor(2^32 / s) + 1.
void set_lap_geometry(GatherArgs *a, uint64_t n, uint64_t s_mod) {
    a->lap_q = static_cast<uint32_t>(n / s_mod);
    a->lap_m = static_cast<uint32_t>(n % s_mod);
    a->div_magic = static_cast<uint32_t>((uint64_t(1) << 32) / s_mod + 1);
}

// Which gather kernel runs, from the path and schedule selections:
//   span     EW_PATH_V256 chosen explicitly: 4-byte elements, s = 2 or 4;
//   tiled    EW_SCHED_TILED, or AUTO where auto_tiled() says so, for s <= 64;
//   laps     AUTO below that, or EW_SCHED_LAPS, once every lap holds a block;
//   oneshot  index order, one block per chunk (n <= 2^32);
//   stride   index order, grid-stride (EW_SCHED_PERSISTENT, or n > 2^32).
GatherKind choose_gather(int e, uint64_t n, uint64_t s_mod) {
    const int path = g_path.load(std::memory_order_relaxed);
    const int sched = g_schedule.load(std::memory_order_relaxed);
    const bool small_n = n <= kOneshotMaxN;
    if (path == EW_PATH_V256 && e == 4 && (s_mod == 2 || s_mod == 4) && small_n) return GatherKind::SPAN;
    if (sched == EW_SCHED_PERSISTENT || !small_n) return GatherKind::STRIDE;
    const bool small_stride = s_mod >= 2 && s_mod <= kMaxLaps;
    const bool tiled = sched == EW_SCHED_TILED || (sched == EW_SCHED_AUTO && auto_tiled(e, s_mod));
    if (small_stride && tiled) return GatherKind::TILED;
    const GatherEntry *laps = e == 4 ? gather_laps_4() : gather_laps_2();
    const uint64_t lap_block = static_cast<uint64_t>(kBlock) * laps->unroll;
    if (sched != EW_SCHED_ONESHOT && small_stride && n / s_mod >= lap_block) return GatherKind::LAPS;
    return GatherKind::ONESHOT;
}

// Span variant: each thread loads the contiguous 8s-element source span of 8
// outputs with 256-bit loads; a scalar head reaches 32-byte output alignment.
GatherLaunch plan_gather_span(const void *in, void *out, uint64_t n, uint64_t s_mod) {
    GatherLaunch gl;
    gl.entry = gather_span_4(static_cast<int64_t>(s_mod));
    gl.args = gather_args(in, out, n, s_mod);
    gl.args.barrett_m = ~uint64_t(0) / n;
    const uintptr_t o = reinterpret_cast<uintptr_t>(out);
    gl.args.head = std::min<int64_t>(static_cast<int64_t>(((32 - o % 32) % 32) / 4), static_cast<int64_t>(n));
    gl.args.nvec = (static_cast<int64_t>(n) - gl.args.head) / 8;
    gl.args.tail0 = gl.args.head + 8 * gl.args.nvec;
    const int64_t per_block = static_cast<int64_t>(kBlock) * gl.entry->unroll;
    gl.grid = clamp_grid((gl.args.nvec + per_block - 1) / per_block);
    gl.path = EW_PATH_V256;
    gl.vec_bytes = 32;
    gl.head = gl.args.head;
    gl.nvec = gl.args.nvec;
    gl.tail = static_cast<int64_t>(n) - gl.args.tail0;
    return gl;
}

// Tiled kernels: P positions of every lap per block, the input span they
// draw from staged in shared memory, rows padded.  On a 16-byte aligned input
// a power-of-two stride (2 to 64) takes the kernel specialised for it; every
// other stride (3 to 63) takes the fixed-stride kernel on any input (its
// shifted instance past a 16-byte boundary), and so do 2-byte elements at
// s = 2, 4 and 8 past a 16-byte boundary; the other powers of two there take
// the general kernel (P a power of two, span up to 20 KiB unless that leaves
// lap runs under 512 bytes).  All stage with 16-byte loads (the launch record
// shows EW_PATH_V128 and vec_bytes 16).
GatherLaunch plan_gather_tiled(int e, const void *in, void *out, uint64_t n, uint64_t s_mod) {
    GatherLaunch gl;
    const GatherEntry *pow2 = e == 4 ? gather_tiled_pow2_4(s_mod) : gather_tiled_pow2_2(s_mod);
    if (pow2 != nullptr && reinterpret_cast<uintptr_t>(in) % 16 == 0) {
        gl.entry = pow2;
        gl.args = gather_args(in, out, n, s_mod);
        gl.args.tile_p = (kTiledPow2SpanBytes / e) / static_cast<uint32_t>(s_mod);
        set_lap_geometry(&gl.args, n, s_mod);
        const uint64_t lap_len = (n + s_mod - 1) / s_mod;
        gl.grid = clamp_grid(static_cast<int64_t>((lap_len + gl.args.tile_p - 1) / gl.args.tile_p));
        gl.path = EW_PATH_V128;
        gl.vec_bytes = 16;
        gl.smem = pow2->smem_bytes;
        gl.block = kTiledPow2Threads;
        gl.schedule = EW_SCHED_TILED;
        gl.nvec = static_cast<int64_t>(n);
        return gl;
    }
    // any element-aligned input: past a 16-byte boundary the shifted instance
    // moves its loads to the boundaries
    const GatherEntry *fixed = gather_tiled_fixed(e, s_mod, reinterpret_cast<uintptr_t>(in) % 16 != 0);
    if (fixed != nullptr) {
        gl.entry = fixed;
        gl.args = gather_args(in, out, n, s_mod);
        gl.args.tile_p = fixed->tile_p;
        gl.args.tile_pitch = fixed->tile_p + fixed_pad_elems(e, static_cast<uint32_t>(s_mod), fixed->tile_p,
                                                             static_cast<uint32_t>(fixed->block));
        set_lap_geometry(&gl.args, n, s_mod);
        const uint64_t lap_len = (n + s_mod - 1) / s_mod;
        gl.grid = clamp_grid(static_cast<int64_t>((lap_len + gl.args.tile_p - 1) / gl.args.tile_p));
        gl.path = EW_PATH_V128;
        gl.vec_bytes = 16;
        gl.smem = static_cast<int32_t>(s_mod * gl.args.tile_pitch * e);
        gl.block = fixed->block;
        gl.schedule = EW_SCHED_TILED;
        gl.nvec = static_cast<int64_t>(n);
        return gl;
    }
    gl.entry = e == 4 ? gather_tiled_4() : gather_tiled_2();
    gl.args = gather_args(in, out, n, s_mod);
    // P: the largest power of two whose span s*P*e stays within
    // kTiledStageBytes, raised until a lap run is kTiledMinRunBytes long.
    // Measured on GB300 at 2^26 (strides 3 to 48, both element sizes): blocks
    // staging 24 KiB or more (8 per SM) ran 9-13% slower than ones staging
    // 12-20 KiB, the shared memory then leaving little of the SM's L1 for
    // loads in flight; runs below 512 bytes made the store phase the limit.
    const uint32_t su = static_cast<uint32_t>(s_mod), eu = static_cast<uint32_t>(e);
    uint32_t log2p = 0;
    while ((2u << log2p) * su * eu <= kTiledStageBytes) ++log2p;
    while ((1u << log2p) * eu < kTiledMinRunBytes) ++log2p;
    gl.args.tile_p = 1u << log2p;
    gl.args.tile_pitch = gl.args.tile_p + tiled_pad_words(su, e, gl.args.tile_p) * (4 / e);
    set_lap_geometry(&gl.args, n, s_mod);
    const uint64_t lap_len = (n + s_mod - 1) / s_mod;
    gl.grid = clamp_grid(static_cast<int64_t>((lap_len + gl.args.tile_p - 1) / gl.args.tile_p));
    gl.path = EW_PATH_V128;  // 16-byte staging loads from each span's first 16-byte boundary
    gl.vec_bytes = 16;
    gl.smem = static_cast<int32_t>(s_mod * gl.args.tile_pitch * e);
    gl.schedule = EW_SCHED_TILED;
    gl.nvec = static_cast<int64_t>(n);
    return gl;
}

// Lap order: block b takes chunk b / s of lap b mod s.
GatherLaunch plan_gather_laps(int e, const void *in, void *out, uint64_t n, uint64_t s_mod) {
    GatherLaunch gl;
    gl.entry = e == 4 ? gather_laps_4() : gather_laps_2();
    gl.args = gather_args(in, out, n, s_mod);
    set_lap_geometry(&gl.args, n, s_mod);
    const uint64_t lap_block = static_cast<uint64_t>(kBlock) * gl.entry->unroll;
    const uint64_t lap_len = (n + s_mod - 1) / s_mod;  // the longest lap
    gl.grid = clamp_grid(static_cast<int64_t>(s_mod * ((lap_len + lap_block - 1) / lap_block)));
    gl.vec_bytes = e;
    gl.schedule = EW_SCHED_LAPS;
    gl.nvec = static_cast<int64_t>(n);
    return gl;
}

// Index order, one block per chunk: (s * i) mod n by Barrett reduction, then
// (s * kBlock) mod n per slot.
GatherLaunch plan_gather_oneshot(int e, const void *in, void *out, uint64_t n, uint64_t s_mod) {
    GatherLaunch gl;
    gl.entry = e == 4 ? gather_oneshot_4() : gather_oneshot_2();
    gl.args = gather_args(in, out, n, s_mod);
    const int64_t per_block = static_cast<int64_t>(kBlock) * gl.entry->unroll;
    gl.grid = clamp_grid((static_cast<int64_t>(n) + per_block - 1) / per_block);
    gl.args.step_mod = (s_mod * static_cast<uint64_t>(kBlock)) % n;  // s_mod < n <= 2^32
    gl.args.barrett_m = ~uint64_t(0) / n;
    gl.vec_bytes = e;
    gl.nvec = static_cast<int64_t>(n);
    return gl;
}

// Index order, grid-stride over SMs x resident blocks: one modular product
// per thread, then (s * T) mod n per slot.
cudaError_t plan_gather_stride(int e, int dev, int sms, const void *in, void *out, uint64_t n, uint64_t s_mod,
                               GatherLaunch *gl) {
    gl->entry = e == 4 ? gather_stride_4() : gather_stride_2();
    gl->args = gather_args(in, out, n, s_mod);
    int occ = 1;
    const cudaError_t ce = blocks_per_sm(dev, gl->entry->kernel, kBlock, 0, &occ);
    if (ce != cudaSuccess) return ce;
    const int64_t per_block = static_cast<int64_t>(kBlock) * gl->entry->unroll;
    gl->grid = clamp_grid(std::min<int64_t>((static_cast<int64_t>(n) + per_block - 1) / per_block,
                                            static_cast<int64_t>(sms) * occ));
    const uint64_t nthr = static_cast<uint64_t>(gl->grid) * kBlock;
    gl->args.step_mod = static_cast<uint64_t>((static_cast<unsigned __int128>(s_mod) * nthr) % n);
    gl->vec_bytes = e;
    gl->schedule = EW_SCHED_PERSISTENT;
    gl->nvec = static_cast<int64_t>(n);
    return cudaSuccess;
}

// Argument checks of a gather call (the pointer-kind check aside).
ew_status check_gather(ew_dtype dt, const void *in, const void *out, int64_t n, int64_t stride) {
    const void *p[2] = {in, out};
    const ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK) return st;
    if (stride <= 0) return EW_ERR_INVALID_VALUE;
    if (n > 0 && overlaps(in, out, n * elem_size(dt))) return EW_ERR_OVERLAP;
    return EW_OK;
}

// The launch a gather call makes (n > 0, arguments checked).  dev < 0: no
// device to ask; the grid-stride kernel's grid, which depends on the SM count
// and occupancy, is then left 0.
cudaError_t plan_gather(int e, const void *in, const void *out, int64_t n, int64_t stride, int dev, int sms,
                        GatherLaunch *gl) {
    const uint64_t un = static_cast<uint64_t>(n);
    const uint64_t s_mod = static_cast<uint64_t>(stride) % un;
    void *o = const_cast<void *>(out);
    switch (choose_gather(e, un, s_mod)) {
        case GatherKind::SPAN: *gl = plan_gather_span(in, o, un, s_mod); break;
        case GatherKind::TILED: *gl = plan_gather_tiled(e, in, o, un, s_mod); break;
        case GatherKind::LAPS: *gl = plan_gather_laps(e, in, o, un, s_mod); break;
        case GatherKind::ONESHOT: *gl = plan_gather_oneshot(e, in, o, un, s_mod); break;
        case GatherKind::STRIDE:
            if (dev >= 0) return plan_gather_stride(e, dev, sms, in, o, un, s_mod, gl);
            gl->entry = e == 4 ? gather_stride_4() : gather_stride_2();
            gl->vec_bytes = e;
            gl->schedule = EW_SCHED_PERSISTENT;
            gl->nvec = n;
            break;
    }
    return cudaSuccess;
}

ew_launch_record record_of(const GatherLaunch &gl) {
    ew_launch_record r{};
    r.launches = 1;
    r.path = gl.path;
    r.vec_bytes = gl.vec_bytes;
    r.grid = gl.grid;
    r.block = gl.block;
    r.smem = gl.smem;
    r.schedule = gl.schedule;
    r.head = gl.head;
    r.nvec = gl.nvec;
    r.tail = gl.tail;
    return r;
}

}  // namespace

bool ew::programmatic_launch() { return g_programmatic.load(std::memory_order_relaxed) != 0; }

// ---------------------------------------------------------------- C ABI

extern "C" {

ew_status ew_add(ew_dtype dt, const void *a, const void *b, void *c, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (!float_dtype(dt)) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[3] = {a, b, c};
    ew_status st = check_common(dt, n, p, 3);
    if (st != EW_OK || n == 0) return st;
    const int64_t bytes = n * elem_size(dt);
    if ((st = check_alias(a, c, bytes)) != EW_OK) return st;
    if ((st = check_alias(b, c, bytes)) != EW_OK) return st;
    return run_stream(OP_ADD, dt, a, b, c, n, 0.0f, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_saxpy(ew_dtype dt, float alpha, const void *x, void *y, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (!float_dtype(dt)) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[2] = {x, y};
    ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK || n == 0) return st;
    if ((st = check_alias(x, y, n * elem_size(dt))) != EW_OK) return st;
    return run_stream(OP_SAXPY, dt, x, y, y, n, alpha, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_saxpy_relu(ew_dtype dt, float alpha, const void *x, void *y, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (!float_dtype(dt)) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[2] = {x, y};
    ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK || n == 0) return st;
    if ((st = check_alias(x, y, n * elem_size(dt))) != EW_OK) return st;
    return run_stream(OP_SAXPY_RELU, dt, x, y, y, n, alpha, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_relu(ew_dtype dt, const void *x, void *y, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (!float_dtype(dt)) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[2] = {x, y};
    ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK || n == 0) return st;
    if ((st = check_alias(x, y, n * elem_size(dt))) != EW_OK) return st;
    // in place, a vector that ReLU leaves unchanged is not stored again
    return run_stream(OP_RELU, dt, x, nullptr, y, n, 0.0f, reinterpret_cast<cudaStream_t>(s), x == y);
}

ew_status ew_add_relu(ew_dtype dt, const void *a, const void *b, void *c, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (!float_dtype(dt)) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[3] = {a, b, c};
    ew_status st = check_common(dt, n, p, 3);
    if (st != EW_OK || n == 0) return st;
    const int64_t bytes = n * elem_size(dt);
    if ((st = check_alias(a, c, bytes)) != EW_OK) return st;
    if ((st = check_alias(b, c, bytes)) != EW_OK) return st;
    return run_stream(OP_ADD_RELU, dt, a, b, c, n, 0.0f, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_select_even_odd(ew_dtype dt, const void *x, void *y, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (dt != EW_I32) return EW_ERR_UNSUPPORTED_DTYPE;
    const void *p[2] = {x, y};
    ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK || n == 0) return st;
    if ((st = check_alias(x, y, n * elem_size(dt))) != EW_OK) return st;
    return run_stream(OP_SELECT, dt, x, nullptr, y, n, 0.0f, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_copy(ew_dtype dt, const void *in, void *out, int64_t n, ew_stream_t s) {
    t_last = ew_launch_record{};
    const void *p[2] = {in, out};
    ew_status st = check_common(dt, n, p, 2);
    if (st != EW_OK || n == 0) return st;
    if ((st = check_alias(in, out, n * elem_size(dt))) != EW_OK) return st;
    if (in == out) return EW_OK;  // nothing to move
    return run_stream(OP_COPY, dt, in, nullptr, out, n, 0.0f, reinterpret_cast<cudaStream_t>(s));
}

ew_status ew_gather_stride(ew_dtype dt, const void *in, void *out, int64_t n, int64_t stride,
                           ew_stream_t s) {
    t_last = ew_launch_record{};
    const void *p[2] = {in, out};
    ew_status st = check_gather(dt, in, out, n, stride);
    if (st != EW_OK || n == 0) return st;
    if (pointer_check_enabled()) {
        if ((st = check_device_pointers(p, 2)) != EW_OK) return st;
    }
    int dev = 0, sms = 0;
    cudaError_t ce = device_info(&dev, &sms);
    if (ce != cudaSuccess) return cuda_fail(ce);
    GatherLaunch gl;
    if ((ce = plan_gather(elem_size(dt), in, out, n, stride, dev, sms, &gl)) != cudaSuccess) return cuda_fail(ce);
    ce = gl.entry->launch(gl.args, gl.grid, reinterpret_cast<cudaStream_t>(s));
    if (ce != cudaSuccess) return cuda_fail(ce);
    t_last = record_of(gl);
    return EW_OK;
}

ew_status ew_gather_plan_query(ew_dtype dt, const void *in, const void *out, int64_t n, int64_t stride,
                               ew_launch_record *out_record) {
    if (out_record == nullptr) return EW_ERR_NULL_POINTER;
    const ew_status st = check_gather(dt, in, out, n, stride);
    if (st != EW_OK) return st;
    *out_record = ew_launch_record{};
    if (n == 0) return EW_OK;
    GatherLaunch gl;
    plan_gather(elem_size(dt), in, out, n, stride, -1, 0, &gl);  // no device: grid-stride grid left 0
    *out_record = record_of(gl);
    return EW_OK;
}

ew_status ew_set_path(ew_path path) {
    const int p = static_cast<int>(path);
    if (p < EW_PATH_AUTO || p > EW_PATH_TMA) return EW_ERR_INVALID_VALUE;
    g_path.store(p, std::memory_order_relaxed);
    return EW_OK;
}

ew_path ew_get_path(void) { return static_cast<ew_path>(g_path.load(std::memory_order_relaxed)); }

ew_status ew_set_schedule(ew_schedule sched) {
    const int v = static_cast<int>(sched);
    if (v < EW_SCHED_AUTO || v > EW_SCHED_TILED) return EW_ERR_INVALID_VALUE;
    g_schedule.store(v, std::memory_order_relaxed);
    return EW_OK;
}

ew_schedule ew_get_schedule(void) {
    return static_cast<ew_schedule>(g_schedule.load(std::memory_order_relaxed));
}

ew_status ew_set_programmatic_launch(int enable) {
    if (enable != 0 && enable != 1) return EW_ERR_INVALID_VALUE;
    g_programmatic.store(enable, std::memory_order_relaxed);
    return EW_OK;
}

int ew_get_programmatic_launch(void) { return g_programmatic.load(std::memory_order_relaxed); }

ew_status ew_set_pointer_check(int enable) {
    if (enable != 0 && enable != 1) return EW_ERR_INVALID_VALUE;
    g_pointer_check.store(enable, std::memory_order_relaxed);
    return EW_OK;
}

ew_status ew_plan_query(ew_dtype dt, const void *const *ptrs, int32_t nptrs, int64_t n, ew_plan *out) {
    if (out == nullptr || ptrs == nullptr) return EW_ERR_NULL_POINTER;
    if (nptrs < 1 || nptrs > 4) return EW_ERR_INVALID_VALUE;
    ew_status st = check_common(dt, n, ptrs, nptrs);
    if (st != EW_OK) return st;
    uintptr_t up[4];
    for (int k = 0; k < nptrs; ++k) up[k] = reinterpret_cast<uintptr_t>(ptrs[k]);
    const int e = elem_size(dt);
    const int path = selected_path();
    ew_plan pl = make_plan(path, e, up, nptrs, n);
    if ((path == EW_PATH_TMA || auto_realign(e, pl, n)) && tma_grid_fits(n, e)) {
        TmaPlan tp;
        if (pl.vec_bytes >= 16) {
            tp = make_tma_plan(make_plan(EW_PATH_V128, e, up, nptrs, n), e, n);
        } else {  // realigning kernel: tiles follow the output, the last pointer
            tp = make_realign_plan(up[nptrs - 1], e, n);
        }
        pl.path = EW_PATH_TMA;
        pl.vec_bytes = 16;
        pl.head = tp.head;
        pl.nvec = tp.ntiles;
        pl.tail = n - tp.rem0;
    }
    *out = pl;
    return EW_OK;
}

ew_status ew_last_launch(ew_launch_record *out) {
    if (out == nullptr) return EW_ERR_NULL_POINTER;
    *out = t_last;
    return EW_OK;
}

const char *ew_status_string(ew_status st) {
    switch (st) {
        case EW_OK: return "EW_OK";
        case EW_ERR_INVALID_VALUE: return "EW_ERR_INVALID_VALUE: bad size, stride, alignment or enum";
        case EW_ERR_NULL_POINTER: return "EW_ERR_NULL_POINTER: null pointer with n > 0";
        case EW_ERR_UNSUPPORTED_DTYPE: return "EW_ERR_UNSUPPORTED_DTYPE: dtype not supported by this operation";
        case EW_ERR_OVERLAP: return "EW_ERR_OVERLAP: output partially overlaps an input";
        case EW_ERR_NOT_DEVICE_POINTER: return "EW_ERR_NOT_DEVICE_POINTER: pointer not accessible by the device";
        case EW_ERR_CUDA: return "EW_ERR_CUDA: CUDA runtime error (see ew_last_cuda_error)";
        case EW_ERR_TIMEOUT: return "EW_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown ew_status";
}

int ew_last_cuda_error(void) { return t_last_cuda_error; }

ew_status ew_device_error(ew_stream_t s, int32_t *code) {
    if (code == nullptr) return EW_ERR_NULL_POINTER;
    cudaError_t e = read_and_clear_device_error(reinterpret_cast<cudaStream_t>(s), code);
    if (e != cudaSuccess) return cuda_fail(e);
    return *code != 0 ? EW_ERR_TIMEOUT : EW_OK;
}

ew_status ew_selftest_bounded_wait(int64_t limit_ns, ew_stream_t s) {
    t_last = ew_launch_record{};
    if (limit_ns < 1 || limit_ns > 10000000000LL) return EW_ERR_INVALID_VALUE;
    cudaError_t e = launch_wait_selftest(static_cast<uint64_t>(limit_ns), reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return cuda_fail(e);
    t_last.launches = 1;
    t_last.grid = 1;
    t_last.block = 32;
    return EW_OK;
}

int ew_version(void) { return 600; }

}  // extern "C"
