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
    } else {
        return ((f >> c) & 1u) ? sc : -sc;
    }
}

}  // namespace qc
