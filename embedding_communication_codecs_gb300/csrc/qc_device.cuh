// qc_device.cuh -- device helpers shared by the libqcodec kernels (sm_103a).
//
// Every arithmetic step that decides a code or a stored float goes through an
// explicit round-to-nearest intrinsic (__fadd_rn, __fsub_rn, __fmul_rn, __fdiv_rn,
// __fmaf_rn), and the library is compiled with -fmad=false, so no operation is
// contracted or reassociated behind the code's back.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qc_internal.h"

namespace qc {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3", SC'11).  Each of the ten rounds takes
// the 32x32->64 products of counter words 0 and 2 with the two round
// multipliers; the new words 0 and 2 are the high halves xor the other counter
// word and a key word, the new words 1 and 3 are the low halves.  The key is
// advanced by the two Weyl constants between rounds; the ten round keys depend
// only on the seed, so the host computes them once per launch (PhiloxKeys) and
// the kernels read them from their constant parameter bank.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys &k) {
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t pA = static_cast<uint64_t>(kMulA) * c.x;  // one wide multiply each
        const uint64_t pB = static_cast<uint64_t>(kMulB) * c.z;
        c = make_uint4(static_cast<uint32_t>(pB >> 32) ^ c.y ^ k.a[r], static_cast<uint32_t>(pB),
                       static_cast<uint32_t>(pA >> 32) ^ c.w ^ k.b[r], static_cast<uint32_t>(pA));
    }
    return c;
}

// The four raw Philox words of elements i0 .. i0+3 (i0 % 4 == 0): counter
// (i0/4 low, i0/4 high, step, 0), key (seed low, seed high).
__device__ __forceinline__ uint4 philox_words(uint64_t i0, uint32_t step, const PhiloxKeys &k) {
    const uint64_t blk = i0 >> 2;
    return philox4x32_10(
        make_uint4(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), step, 0u), k);
}

// Four uniform draws u in [0, 1) for elements i0 .. i0+3 (i0 % 4 == 0):
// counter (i0/4 low, i0/4 high, step, 0), key (seed low, seed high),
// u = (word >> 8) * 2^-24, exact in binary32.
__device__ __forceinline__ void uniform4(uint64_t i0, uint32_t step, const PhiloxKeys &k,
                                         float u[4]) {
    const uint64_t blk = i0 >> 2;
    const uint4 r = philox4x32_10(
        make_uint4(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), step, 0u), k);
    u[0] = __fmul_rn(__uint2float_rn(r.x >> 8), 0x1p-24f);
    u[1] = __fmul_rn(__uint2float_rn(r.y >> 8), 0x1p-24f);
    u[2] = __fmul_rn(__uint2float_rn(r.z >> 8), 0x1p-24f);
    u[3] = __fmul_rn(__uint2float_rn(r.w >> 8), 0x1p-24f);
}

// The single draw u for element i (the same value uniform4 gives it).
__device__ __forceinline__ float uniform1(uint64_t i, uint32_t step, const PhiloxKeys &k) {
    const uint64_t blk = i >> 2;
    const uint4 r = philox4x32_10(
        make_uint4(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32), step, 0u), k);
    const uint32_t c = static_cast<uint32_t>(i & 3u);
    const uint32_t w = c == 0 ? r.x : c == 1 ? r.y : c == 2 ? r.z : r.w;
    return __fmul_rn(__uint2float_rn(w >> 8), 0x1p-24f);
}

// ---------------------------------------------------------------------------
// Integer helpers without conversion instructions.

// rint(t) for 0 <= t < 2^22, ties to even: adding 1.5 * 2^23 leaves the rounded
// integer in the low mantissa bits.
__device__ __forceinline__ uint32_t rint_small(float t) {
    return __float_as_uint(__fadd_rn(t, 12582912.0f)) - 0x4B400000u;
}

// Exact binary32 value of an integer 0 <= q < 2^23.
__device__ __forceinline__ float small_uint_to_float(uint32_t q) {
    return __fsub_rn(__uint_as_float(0x4B000000u | q), 8388608.0f);
}

__device__ __forceinline__ float positive_zero(float r) { return r == 0.0f ? 0.0f : r; }

// ---------------------------------------------------------------------------
// Warp butterflies.  XOR butterflies leave the same value in every lane; the
// operations used are commutative, so partner lanes compute identical results.

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Double-word (hi, lo) accumulation.  two_sum returns the exact error of a+b.
__device__ __forceinline__ float two_sum(float a, float b, float &err) {
    const float s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    const float ap = __fsub_rn(s, bp);
    err = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
    return s;
}

struct DWord {
    float hi, lo;
};

__device__ __forceinline__ DWord dw_add(DWord a, DWord b) {
    float e;
    const float s = two_sum(a.hi, b.hi, e);
    return DWord{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

__device__ __forceinline__ DWord dw_add(DWord a, float x) {
    float e;
    const float s = two_sum(a.hi, x, e);
    return DWord{s, __fadd_rn(a.lo, e)};
}

__device__ __forceinline__ DWord warp_sum(DWord v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        DWord p{__shfl_xor_sync(kFull, v.hi, o), __shfl_xor_sync(kFull, v.lo, o)};
        v = dw_add(v, p);
    }
    return v;
}

// fl((hi + lo) / d) for a small positive integer d held exactly as a float:
// quotient of hi, exact remainder by fma, then the remainder's share.
__device__ __forceinline__ float dw_div(DWord v, float d) {
    const float q0 = __fdiv_rn(v.hi, d);
    const float r = __fadd_rn(__fmaf_rn(-q0, d, v.hi), v.lo);
    return __fadd_rn(q0, __fdiv_rn(r, d));
}

// ---------------------------------------------------------------------------
// Packing: each lane holds the 4 codes of its 4 consecutive elements as a
// (4*BITS)-bit field, element 0 lowest.  Lanes 8/BITS apart hold consecutive
// fields of one 32-bit word; shuffles gather the word into the lowest of them.
template <int BITS>
__device__ __forceinline__ uint32_t gather_word(uint32_t field) {
    constexpr int kLanesPerWord = 8 / BITS;
#pragma unroll
    for (int off = 1; off < kLanesPerWord; off <<= 1)
        field |= __shfl_down_sync(kFull, field, off) << (off * 4 * BITS);
    return field;
}

template <int BITS>
__device__ __forceinline__ bool stores_word(int lane) {
    return (lane & (8 / BITS - 1)) == 0;
}

// ---------------------------------------------------------------------------
// Loads of four consecutive gradient elements as fp32.

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

template <typename TIn>
struct GradLoad;

template <>
struct GradLoad<float> {
    // full: four elements in range, 16-byte aligned
    static __device__ __forceinline__ float4 full(const float *g, uint64_t i) {
        return __ldcs(reinterpret_cast<const float4 *>(g + i));
    }
    static __device__ __forceinline__ float one(const float *g, uint64_t i) { return __ldcs(g + i); }
};

__device__ __forceinline__ float4 unpack_bf16x4(uint2 v) {
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
}

template <>
struct GradLoad<uint16_t> {
    static __device__ __forceinline__ float4 full(const uint16_t *g, uint64_t i) {
        return unpack_bf16x4(__ldcs(reinterpret_cast<const uint2 *>(g + i)));
    }
    static __device__ __forceinline__ float one(const uint16_t *g, uint64_t i) {
        return bf16_bits_to_float(__ldcs(reinterpret_cast<const unsigned short *>(g + i)));
    }
};

__device__ __forceinline__ float get(const float4 &v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__device__ __forceinline__ void set(float4 &v, int j, float x) {
    if (j == 0) v.x = x;
    else if (j == 1) v.y = x;
    else if (j == 2) v.z = x;
    else v.w = x;
}

}  // namespace qc
