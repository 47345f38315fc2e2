// qc_exact_norm.cuh -- the exactly rounded L2 norm of a bucket, for the rare
// buckets where the double-word estimate cannot decide the rounding.
//
// QSGD scales a bucket by its L2 norm ("Quantization for Communication",
// Quantized SGD Algorithms).  The norm is the binary32 value nearest (ties to
// even) to the square root of the exact sum of the squares.  The fast path
// (Stats<kQsgd> and Finish<kQsgd> in qc_encode_math.cuh) estimates it from a
// double-word sum with a proven error bound and takes this path only when the
// estimate lies within that bound of a rounding boundary, or outside the range
// where the bound holds.
//
// Here every square is added exactly into a wide fixed-point integer: a
// binary32 x = m * 2^e (integer m < 2^24, e >= -149) has x^2 = m^2 * 2^(2e), an
// integer multiple of 2^-300, so the sum is held as an unsigned integer in units
// of 2^-300 in kWideLimbs 32-bit limbs (squares are below 2^256 and a bucket
// holds at most 2^24 of them, so the sum stays below 2^280, i.e. 2^580 units).
// The rounding is decided by comparing that integer with the exact squares of the midpoints around a candidate: for f = m * 2^e the upper
// midpoint is (2m + 1) * 2^(e-1), whose square is (2m + 1)^2 * 2^(2e+298) units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qc {

constexpr int kWideLimbs = 20;  // 640 bits

struct WideSum {
    uint32_t w[kWideLimbs];
};

__device__ __forceinline__ void wide_zero(WideSum &a) {
#pragma unroll
    for (int i = 0; i < kWideLimbs; ++i) a.w[i] = 0u;
}

// a += v * 2^pos for v < 2^64: v * 2^(pos mod 32) spans three limbs from limb
// pos / 32, then the carry runs up.
__device__ __forceinline__ void wide_add_shifted(WideSum &a, uint64_t v, uint32_t pos) {
    const uint32_t k = pos >> 5, sh = pos & 31u;
    uint32_t part[3];
    part[0] = static_cast<uint32_t>(v << sh);
    part[1] = static_cast<uint32_t>(sh ? (v >> (32u - sh)) : (v >> 32));
    part[2] = sh ? static_cast<uint32_t>(v >> (64u - sh)) : 0u;
    uint64_t carry = 0;
    for (uint32_t i = k; i < static_cast<uint32_t>(kWideLimbs); ++i) {
        const uint32_t add = (i - k < 3u) ? part[i - k] : 0u;
        if (i - k >= 3u && carry == 0) break;
        const uint64_t s = static_cast<uint64_t>(a.w[i]) + add + carry;
        a.w[i] = static_cast<uint32_t>(s);
        carry = s >> 32;
    }
}

// a += x^2 in units of 2^-300; non-finite x is skipped (its square has no
// place in a finite sum; the codes of such a bucket are unspecified).
__device__ __forceinline__ void wide_add_square(WideSum &a, float x) {
    const uint32_t b = __float_as_uint(x);
    const uint32_t ex = (b >> 23) & 0xFFu;
    if (ex == 0xFFu) return;
    uint32_t m = b & 0x7FFFFFu;
    int e = -149;
    if (ex) {
        m |= 0x800000u;
        e = static_cast<int>(ex) - 150;
    }
    if (m == 0u) return;
    wide_add_shifted(a, static_cast<uint64_t>(m) * m, static_cast<uint32_t>(2 * e + 300));
}

// a += b (both normalised).
__device__ __forceinline__ void wide_add(WideSum &a, const WideSum &b) {
    uint64_t carry = 0;
#pragma unroll
    for (int i = 0; i < kWideLimbs; ++i) {
        const uint64_t s = static_cast<uint64_t>(a.w[i]) + b.w[i] + carry;
        a.w[i] = static_cast<uint32_t>(s);
        carry = s >> 32;
    }
}

// Butterfly sum over the 32 lanes of the warp: every lane ends with the total.
__device__ __forceinline__ void wide_warp_sum(WideSum &a) {
    for (int o = 16; o > 0; o >>= 1) {
        WideSum b;
#pragma unroll
        for (int i = 0; i < kWideLimbs; ++i) b.w[i] = __shfl_xor_sync(0xffffffffu, a.w[i], o);
        wide_add(a, b);
    }
}

// Sign of a - v * 2^pos (v < 2^64): -1, 0 or +1.
__device__ __forceinline__ int wide_cmp_shifted(const WideSum &a, uint64_t v, uint32_t pos) {
    WideSum b;
    wide_zero(b);
    wide_add_shifted(b, v, pos);
    for (int i = kWideLimbs - 1; i >= 0; --i)
        if (a.w[i] != b.w[i]) return a.w[i] > b.w[i] ? 1 : -1;
    return 0;
}

// The binary32 value nearest (ties to even) to sqrt(a * 2^-300).
__device__ __forceinline__ float wide_sqrt_f32(const WideSum &a) {
    int t = kWideLimbs - 1;
    while (t >= 0 && a.w[t] == 0u) --t;
    if (t < 0) return 0.0f;
    // candidate: the square root of the top 96 bits, in binary64, rounded to binary32
    double v = static_cast<double>(a.w[t]);
    if (t >= 1) v = v * 4294967296.0 + static_cast<double>(a.w[t - 1]);
    if (t >= 2) v = v * 4294967296.0 + static_cast<double>(a.w[t - 2]);
    const int low = t >= 2 ? t - 2 : 0;  // v counts units of 2^(32 low - 300), an even power
    float f = __double2float_rn(ldexp(sqrt(v), (32 * low - 300) / 2));
    if (!(f <= 3.4028234663852886e38f)) f = 3.4028234663852886e38f;  // checked against its upper midpoint
    if (f < 1.401298464324817e-45f) f = 1.401298464324817e-45f;      // a >= 4 units: the root is >= 2^-149
    // move f until a lies between the squares of its two midpoints
    for (int iter = 0; iter < 4; ++iter) {
        const uint32_t fb = __float_as_uint(f);
        const uint32_t ex = fb >> 23;
        uint32_t m = fb & 0x7FFFFFu;
        int e = -149;
        if (ex) {
            m |= 0x800000u;
            e = static_cast<int>(ex) - 150;
        }
        if (m == 0u) return f;
        // upper midpoint (2m + 1) 2^(e-1)
        const uint64_t mu = 2ull * m + 1ull;
        const int cu = wide_cmp_shifted(a, mu * mu, static_cast<uint32_t>(2 * e + 298));
        if (cu > 0 || (cu == 0 && (m & 1u))) {  // above it, or on it with f odd
            if (fb == 0x7F7FFFFFu) return __uint_as_float(0x7F800000u);  // rounds to 2^128
            f = __uint_as_float(fb + 1u);
            continue;
        }
        // lower midpoint: (2m - 1) 2^(e-1), or (4m - 1) 2^(e-2) at the bottom of a binade
        int cl;
        if (m == 0x800000u && ex > 1u) {
            const uint64_t ml = 4ull * m - 1ull;
            cl = wide_cmp_shifted(a, ml * ml, static_cast<uint32_t>(2 * e + 296));
        } else {
            const uint64_t ml = 2ull * m - 1ull;
            cl = wide_cmp_shifted(a, ml * ml, static_cast<uint32_t>(2 * e + 298));
        }
        if (cl < 0 || (cl == 0 && (m & 1u))) {  // below it, or on it with f odd
            f = __uint_as_float(fb - 1u);
            continue;
        }
        return f;
    }
    return f;
}

}  // namespace qc
