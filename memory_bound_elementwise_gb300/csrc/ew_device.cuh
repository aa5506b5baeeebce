// ew_device.cuh -- device-side building blocks: raw vector memory access and
// the per-element operators, all written as explicit PTX so that the rounding
// of every operation is visible in the source.
//
// Memory access: one access moves VB bytes of raw bits (VB = 32, 16, 8, 4 or
// 2).  32-byte accesses use the 256-bit ld/st forms of the sm_100 family.
// Loads and stores skip L1 allocation: every byte is touched exactly once.
//
// Operators work on 32-bit words (one binary32, or two packed 16-bit
// elements) and on single 16-bit elements (for 2-byte scalar heads and tails).
#pragma once

#include <cstdint>

namespace ew {

// ---------------------------------------------------------------- launches
//
// First statements of every kernel: wait until the grid before this one on
// the stream has completed and its writes are visible (a no-op when there is
// none or when launched without programmatic serialisation), then allow the
// grid after this one to be scheduled.

__device__ __forceinline__ void enter_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- vectors

template <int VB> struct Vec;
template <> struct Vec<32> { uint32_t w[8]; static constexpr int kWords = 8; };
template <> struct Vec<16> { uint32_t w[4]; static constexpr int kWords = 4; };
template <> struct Vec<8>  { uint32_t w[2]; static constexpr int kWords = 2; };
template <> struct Vec<4>  { uint32_t w[1]; static constexpr int kWords = 1; };
template <> struct Vec<2>  { uint16_t h;    static constexpr int kWords = 0; };

template <int VB> __device__ __forceinline__ Vec<VB> ld(const void *p);
template <int VB> __device__ __forceinline__ void st(void *p, const Vec<VB> &v);

template <> __device__ __forceinline__ Vec<32> ld<32>(const void *p) {
    Vec<32> v;
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]),
                   "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}
template <> __device__ __forceinline__ Vec<16> ld<16>(const void *p) {
    Vec<16> v;
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
    return v;
}
template <> __device__ __forceinline__ Vec<8> ld<8>(const void *p) {
    Vec<8> v;
    asm volatile("ld.global.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
                 : "=r"(v.w[0]), "=r"(v.w[1]) : "l"(p));
    return v;
}
template <> __device__ __forceinline__ Vec<4> ld<4>(const void *p) {
    Vec<4> v;
    asm volatile("ld.global.L1::no_allocate.b32 %0, [%1];" : "=r"(v.w[0]) : "l"(p));
    return v;
}
template <> __device__ __forceinline__ Vec<2> ld<2>(const void *p) {
    Vec<2> v;
    asm volatile("ld.global.L1::no_allocate.b16 %0, [%1];" : "=h"(v.h) : "l"(p));
    return v;
}

template <> __device__ __forceinline__ void st<32>(void *p, const Vec<32> &v) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]),
                    "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}
template <> __device__ __forceinline__ void st<16>(void *p, const Vec<16> &v) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
}
template <> __device__ __forceinline__ void st<8>(void *p, const Vec<8> &v) {
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1,%2};"
                 :: "l"(p), "r"(v.w[0]), "r"(v.w[1]) : "memory");
}
template <> __device__ __forceinline__ void st<4>(void *p, const Vec<4> &v) {
    asm volatile("st.global.L1::no_allocate.b32 [%0], %1;" :: "l"(p), "r"(v.w[0]) : "memory");
}
template <> __device__ __forceinline__ void st<2>(void *p, const Vec<2> &v) {
    asm volatile("st.global.L1::no_allocate.b16 [%0], %1;" :: "l"(p), "h"(v.h) : "memory");
}

// ---------------------------------------------------------------- arithmetic

__device__ __forceinline__ uint32_t add_f32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t add_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint16_t add_f16(uint16_t a, uint16_t b) {
    uint16_t d;
    asm("add.rn.f16 %0, %1, %2;" : "=h"(d) : "h"(a), "h"(b));
    return d;
}
__device__ __forceinline__ uint16_t add_bf16(uint16_t a, uint16_t b) {
    uint16_t d;
    asm("add.rn.bf16 %0, %1, %2;" : "=h"(d) : "h"(a), "h"(b));
    return d;
}
__device__ __forceinline__ float fma_f32(float a, float x, float y) {
    float d;
    asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(x), "f"(y));
    return d;
}
// binary16 <-> binary32 (widening is exact)
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}
__device__ __forceinline__ uint16_t f32_to_f16(float f) {
    uint16_t h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}
// packs round(hi) into bits 31..16 and round(lo) into bits 15..0
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// bfloat16 is the upper half of binary32: widening is a shift
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ReLU on raw bits: negative non-NaN values (and -0) become +0; everything
// else (positive values, +0, NaN of either sign) is kept bit for bit.
__device__ __forceinline__ uint32_t relu_b32(uint32_t u) {
    const bool neg = (u >> 31) != 0u;
    const bool nan = (u & 0x7fffffffu) > 0x7f800000u;
    return (neg && !nan) ? 0u : u;
}
template <uint32_t kInfBits>  // 0x7c00 for binary16, 0x7f80 for bfloat16
__device__ __forceinline__ uint16_t relu_b16(uint16_t h) {
    const bool neg = (h & 0x8000u) != 0u;
    const bool nan = (h & 0x7fffu) > kInfBits;
    return (neg && !nan) ? static_cast<uint16_t>(0) : h;
}
template <uint32_t kInfBits>
__device__ __forceinline__ uint32_t relu_b16x2(uint32_t w) {
    const uint32_t lo = relu_b16<kInfBits>(static_cast<uint16_t>(w & 0xffffu));
    const uint32_t hi = relu_b16<kInfBits>(static_cast<uint16_t>(w >> 16));
    return lo | (hi << 16);
}

// ---------------------------------------------------------------- operators
//
// Each operator has
//   kIn      number of input arrays (1 or 2)
//   kElem    element size in bytes
//   word(...)  one 32-bit word of output from the matching input words
//   half(...)  one 16-bit element (only for kElem == 2)

struct OpAddF32 {
    static constexpr int kIn = 2, kElem = 4;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const { return add_f32(a, b); }
    __device__ __forceinline__ uint16_t half(uint16_t, uint16_t) const { return 0; }
};
struct OpAddF16 {
    static constexpr int kIn = 2, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const { return add_f16x2(a, b); }
    __device__ __forceinline__ uint16_t half(uint16_t a, uint16_t b) const { return add_f16(a, b); }
};
struct OpAddBF16 {
    static constexpr int kIn = 2, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const { return add_bf16x2(a, b); }
    __device__ __forceinline__ uint16_t half(uint16_t a, uint16_t b) const { return add_bf16(a, b); }
};

// SAXPY: inputs are (x, y); output is written over y.
struct OpSaxpyF32 {
    static constexpr int kIn = 2, kElem = 4;
    float alpha;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t y) const {
        return __float_as_uint(fma_f32(alpha, __uint_as_float(x), __uint_as_float(y)));
    }
    __device__ __forceinline__ uint16_t half(uint16_t, uint16_t) const { return 0; }
};
struct OpSaxpyF16 {
    static constexpr int kIn = 2, kElem = 2;
    float alpha;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t y) const {
        const float lo = fma_f32(alpha, f16_to_f32(x & 0xffffu), f16_to_f32(y & 0xffffu));
        const float hi = fma_f32(alpha, f16_to_f32(x >> 16), f16_to_f32(y >> 16));
        return f32x2_to_f16x2(hi, lo);
    }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t y) const {
        return f32_to_f16(fma_f32(alpha, f16_to_f32(x), f16_to_f32(y)));
    }
};
struct OpSaxpyBF16 {
    static constexpr int kIn = 2, kElem = 2;
    float alpha;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t y) const {
        const float lo = fma_f32(alpha, __uint_as_float(x << 16), __uint_as_float(y << 16));
        const float hi = fma_f32(alpha, __uint_as_float(x & 0xffff0000u),
                                 __uint_as_float(y & 0xffff0000u));
        return f32x2_to_bf16x2(hi, lo);
    }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t y) const {
        return f32_to_bf16(fma_f32(alpha, bf16_to_f32(x), bf16_to_f32(y)));
    }
};

struct OpReluF32 {
    static constexpr int kIn = 1, kElem = 4;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t) const { return relu_b32(x); }
    __device__ __forceinline__ uint16_t half(uint16_t, uint16_t) const { return 0; }
};
struct OpReluF16 {
    static constexpr int kIn = 1, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t) const { return relu_b16x2<0x7c00u>(x); }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t) const { return relu_b16<0x7c00u>(x); }
};
struct OpReluBF16 {
    static constexpr int kIn = 1, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t) const { return relu_b16x2<0x7f80u>(x); }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t) const { return relu_b16<0x7f80u>(x); }
};

// Fused bias add + ReLU: C = max(A + B, 0) with the sum rounded first, i.e.
// exactly relu(add(A, B)) in one pass (12 bytes per binary32 element instead
// of 12 + 8 for the two separate passes).
struct OpAddReluF32 {
    static constexpr int kIn = 2, kElem = 4;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const { return relu_b32(add_f32(a, b)); }
    __device__ __forceinline__ uint16_t half(uint16_t, uint16_t) const { return 0; }
};
struct OpAddReluF16 {
    static constexpr int kIn = 2, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const {
        return relu_b16x2<0x7c00u>(add_f16x2(a, b));
    }
    __device__ __forceinline__ uint16_t half(uint16_t a, uint16_t b) const {
        return relu_b16<0x7c00u>(add_f16(a, b));
    }
};
struct OpAddReluBF16 {
    static constexpr int kIn = 2, kElem = 2;
    __device__ __forceinline__ uint32_t word(uint32_t a, uint32_t b) const {
        return relu_b16x2<0x7f80u>(add_bf16x2(a, b));
    }
    __device__ __forceinline__ uint16_t half(uint16_t a, uint16_t b) const {
        return relu_b16<0x7f80u>(add_bf16(a, b));
    }
};

// Fused SAXPY + ReLU: y = max(fmaf(alpha, x, y), 0) with the fma rounded
// first, i.e. exactly relu(saxpy(x, y)) in one pass (12 bytes per binary32
// element instead of 12 + 8).
template <class Saxpy, class Relu>
struct OpSaxpyReluOf {
    static constexpr int kIn = 2, kElem = Saxpy::kElem;
    float alpha;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t y) const {
        return Relu{}.word(Saxpy{alpha}.word(x, y), 0u);
    }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t y) const {
        return Relu{}.half(Saxpy{alpha}.half(x, y), 0);
    }
};
using OpSaxpyReluF32 = OpSaxpyReluOf<OpSaxpyF32, OpReluF32>;
using OpSaxpyReluF16 = OpSaxpyReluOf<OpSaxpyF16, OpReluF16>;
using OpSaxpyReluBF16 = OpSaxpyReluOf<OpSaxpyBF16, OpReluBF16>;

// Even/odd select on 32-bit two's complement integers: y = x even ? 2x : x + 1
// (CUDA-MODE lecture notes §6: the divergent if/else and its branch-free
// rewrite compute the same thing).  Written without a branch: x + (odd ? 1 : x),
// wrapping modulo 2^32.
struct OpSelectEvenOddI32 {
    static constexpr int kIn = 1, kElem = 4;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t) const {
        const uint32_t odd = x & 1u;
        return x + (odd ? 1u : x);
    }
    __device__ __forceinline__ uint16_t half(uint16_t, uint16_t) const { return 0; }
};

template <int E>
struct OpCopy {
    static constexpr int kIn = 1, kElem = E;
    __device__ __forceinline__ uint32_t word(uint32_t x, uint32_t) const { return x; }
    __device__ __forceinline__ uint16_t half(uint16_t x, uint16_t) const { return x; }
};

// Operators whose output can equal their only input bit for bit; for such an
// operator computed in place, a vector whose result equals what is already in
// memory need not be stored.
template <class Op> struct MaySkipUnchanged { static constexpr bool value = false; };
template <> struct MaySkipUnchanged<OpReluF32> { static constexpr bool value = true; };
template <> struct MaySkipUnchanged<OpReluF16> { static constexpr bool value = true; };
template <> struct MaySkipUnchanged<OpReluBF16> { static constexpr bool value = true; };

template <int VB>
__device__ __forceinline__ bool same_bits(const Vec<VB> &x, const Vec<VB> &y) {
    if constexpr (VB == 2) {
        return x.h == y.h;
    } else {
        uint32_t diff = 0;
#pragma unroll
        for (int k = 0; k < Vec<VB>::kWords; ++k) diff |= x.w[k] ^ y.w[k];
        return diff == 0;
    }
}

// Apply an operator to a whole vector.
template <class Op, int VB>
__device__ __forceinline__ Vec<VB> apply(const Op &op, const Vec<VB> &a, const Vec<VB> &b) {
    Vec<VB> c;
    if constexpr (VB == 2) {
        c.h = op.half(a.h, b.h);
    } else {
#pragma unroll
        for (int k = 0; k < Vec<VB>::kWords; ++k) c.w[k] = op.word(a.w[k], b.w[k]);
    }
    return c;
}

// One element at byte offset `off` (scalar heads and tails).
template <class Op>
__device__ __forceinline__ void apply_one(const Op &op, const char *in0, const char *in1,
                                          char *out, int64_t off) {
    if constexpr (Op::kElem == 4) {
        const uint32_t a = ld<4>(in0 + off).w[0];
        const uint32_t b = (Op::kIn == 2) ? ld<4>(in1 + off).w[0] : 0u;
        Vec<4> c;
        c.w[0] = op.word(a, b);
        st<4>(out + off, c);
    } else {
        const uint16_t a = ld<2>(in0 + off).h;
        const uint16_t b = (Op::kIn == 2) ? ld<2>(in1 + off).h : static_cast<uint16_t>(0);
        Vec<2> c;
        c.h = op.half(a, b);
        st<2>(out + off, c);
    }
}

}  // namespace ew
