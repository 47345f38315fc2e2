// qc_decode_math.cuh -- branch-free dequantization of packed codes, shared by
// the decode kernels.
//
// "Quantization for Communication", "Quantization Schemes" (x ~ q * scale + min)
// and "Quantized SGD Algorithms" (TernGrad {-1, 0, +1} times a scale; SignSGD).
// A code c < 2^23 becomes an exact binary32 value through the bit pattern of
// 2^23 + c minus 2^23 (no conversion instruction); the ternary value
// (c - 1) * s is one fused multiply-add fma(c, s, -s), exact for c in 0..3
// because (c - 1) * s is representable; the sign value is a select.
#pragma once

#include "qc_device.cuh"
#include "qc_internal.h"

namespace qc {

// Exact float value of code c (0..3) of a 4*BITS-bit field f (code 0 lowest).
template <int BITS>
__device__ __forceinline__ float code_value(uint32_t f, int c) {
    uint32_t m;
    if constexpr (BITS == 8) {
        m = __byte_perm(f, 0x4B000000u, 0x7540u | static_cast<uint32_t>(c));
    } else {
        m = ((f >> (c * BITS)) & ((1u << BITS) - 1u)) | 0x4B000000u;
    }
    return __fsub_rn(__uint_as_float(m), 8388608.0f);
}

// Dequantized value of code c of field f with the bucket's scale / offset.
template <int SCHEME, int BITS>
__device__ __forceinline__ float dequant_code(uint32_t f, int c, float sc, float of) {
    if constexpr (SCHEME == kUniform) {
        return __fmaf_rn(code_value<BITS>(f, c), sc, of);
    } else if constexpr (SCHEME == kTernary) {
        return __fmaf_rn(code_value<BITS>(f, c), sc, -sc);
    } else if constexpr (SCHEME == kLog) {
        // sign bit over the level index j: +-fl(s * 2^(j - J)), the power of two
        // built from its exponent bits (the level table), 0 for j = 0
        constexpr uint32_t J = (1u << (BITS - 1)) - 1u;
        const uint32_t code = (f >> (c * BITS)) & ((1u << BITS) - 1u);
        const uint32_t lvl = code & J;
        const float mag = lvl ? __fmul_rn(sc, __uint_as_float((lvl + 127u - J) << 23)) : 0.0f;
        return __uint_as_float(__float_as_uint(mag) | ((code << (32 - BITS)) & 0x80000000u));
    } else if constexpr (SCHEME == kQsgd) {
        // sign bit over the level: +-fl(level * unit), the sign set by OR
        const uint32_t code = (f >> (c * BITS)) & ((1u << BITS) - 1u);
        const uint32_t lvl = code & ((1u << (BITS - 1)) - 1u);
        const float mag = __fmul_rn(__fsub_rn(__uint_as_float(lvl | 0x4B000000u), 8388608.0f), sc);
        return __uint_as_float(__float_as_uint(mag) | ((code << (32 - BITS)) & 0x80000000u));
    } else {
        return ((f >> c) & 1u) ? sc : -sc;
    }
}

// acc + (dequantized code c of field f), rounded once as fl(acc + d).  The
// ternary value d = (c - 1) * s is exact, so fl(acc + d) is the single rounding
// of fma(c - 1, s, acc); c - 1 comes from the bit pattern of 2^23 + c minus
// 2^23 + 1.  Uniform values are themselves rounded and need the separate add.
template <int SCHEME, int BITS>
__device__ __forceinline__ float accumulate_code(float acc, uint32_t f, int c, float sc, float of) {
    if constexpr (SCHEME == kTernary) {
        const uint32_t m = ((f >> (c * BITS)) & ((1u << BITS) - 1u)) | 0x4B000000u;
        return __fmaf_rn(__fsub_rn(__uint_as_float(m), 8388609.0f), sc, acc);
    } else {
        return __fadd_rn(acc, dequant_code<SCHEME, BITS>(f, c, sc, of));
    }
}

// The codes of 16 consecutive elements of one worker, read from shared memory
// as 2 * BITS bytes (16-byte, 8-byte, 4-byte or 2-byte load).
template <int BITS>
__device__ __forceinline__ void load_codes16(const unsigned char *src, uint32_t (&f)[4]) {
    if constexpr (BITS == 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else if constexpr (BITS == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(src);
        f[0] = v.x; f[1] = v.y; f[2] = 0u; f[3] = 0u;
    } else if constexpr (BITS == 2) {
        f[0] = *reinterpret_cast<const uint32_t *>(src); f[1] = f[2] = f[3] = 0u;
    } else {
        f[0] = *reinterpret_cast<const unsigned short *>(src); f[1] = f[2] = f[3] = 0u;
    }
}

// acc + the dequantized code c (0..15) of a 16-code group.
template <int SCHEME, int BITS>
__device__ __forceinline__ float accumulate16(float acc, const uint32_t (&f)[4], int c, float sc,
                                              float of) {
    constexpr int kPerWord = 32 / BITS;
    return accumulate_code<SCHEME, BITS>(acc, f[c / kPerWord], c % kPerWord, sc, of);
}

// ---------------------------------------------------- packed pairs (f32x2)
//
// Two fp32 lanes in one 64-bit register, low half first: add.rn.f32x2 and
// fma.rn.f32x2 round each half exactly as the scalar instructions would, in one
// issue slot for both.

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Sixteen ternary codes of one word f (code c in bits 2c, 2c+1) accumulated into
// eight packed pairs: acc = fl(acc + (c - 1) * s) per element.  Code j of a
// half word h becomes an exact float without shifting it down: (h & 3 << 2j)
// OR'd under the exponent of 2^(23 - 2j) is 2^(23 - 2j) + c, so subtracting
// 2^(23 - 2j) + 1 (exact) gives c - 1, and (c - 1) * s is exact, so one fma
// rounds acc + d once, as the scalar accumulate_code does.  The exponent
// fields ex[j] = (150 - 2j) << 23 and the packed biases k2[i] = -(2^(23 - 2j) +
// 1) for j = 2i, 2i + 1 come in registers: with the exponent an immediate as
// well as the mask, the mask-and-merge would take two logic operations.
__device__ __forceinline__ void accumulate_ternary16(unsigned long long (&acc)[8], uint32_t f,
                                                     unsigned long long s2, const uint32_t (&ex)[8],
                                                     const unsigned long long (&k2)[4]) {
    const uint32_t half[2] = {f, f >> 16};  // the masks ignore the other half's bits
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint32_t h = half[p >> 2];
        const int j0 = 2 * (p & 3), j1 = j0 + 1;
        const float m0 = __uint_as_float((h & (3u << (2 * j0))) | ex[j0]);
        const float m1 = __uint_as_float((h & (3u << (2 * j1))) | ex[j1]);
        acc[p] = fma2(add2(pack2(m0, m1), k2[p & 3]), s2, acc[p]);
    }
}

// The 4*BITS-bit field of the four codes of tile element e (e % 4 == 0) of one
// worker: from the stage when staged, else from global memory (tile tail).
template <int BITS>
__device__ __forceinline__ uint32_t field4(const unsigned char *wstage, const uint32_t *wglob,
                                           uint32_t e, uint32_t staged_bytes) {
    const uint32_t byte = (e * BITS) / 8u;
    if constexpr (BITS == 8) {
        return byte + 4u <= staged_bytes ? *reinterpret_cast<const uint32_t *>(wstage + byte)
                                         : __ldcs(wglob + e / 4u);
    } else if constexpr (BITS == 4) {
        return byte + 2u <= staged_bytes
                   ? *reinterpret_cast<const unsigned short *>(wstage + byte)
                   : __ldcs(reinterpret_cast<const unsigned short *>(wglob) + e / 4u);
    } else if constexpr (BITS == 2) {
        return byte < staged_bytes ? wstage[byte]
                                   : __ldcs(reinterpret_cast<const unsigned char *>(wglob) + e / 4u);
    } else {
        const uint32_t b = byte < staged_bytes
                               ? wstage[byte]
                               : __ldcs(reinterpret_cast<const unsigned char *>(wglob) + e / 8u);
        return (b >> ((e & 4u) ? 4u : 0u)) & 0xFu;
    }
}

}  // namespace qc
