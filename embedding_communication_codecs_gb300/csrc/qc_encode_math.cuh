// qc_encode_math.cuh -- per-bucket statistics, bucket parameters, per-element
// quantization and the slot-level quantize/store step shared by the encode
// kernels (direct and TMA-pipelined).
//
// "Quantization for Communication", "Quantization Schemes" (uniform min/max:
// scale = (max - min) / (2^bits - 1), q = round((x - min) / scale), x ~ q * scale
// + min; stochastic rounding takes the floor with probability 1 - frac and the
// ceiling with probability frac), "Quantized SGD Algorithms" (TernGrad
// {-1, 0, +1} with a scale; SignSGD), "Error Feedback for Quantization"
// (e = e + g; q = quantize(e); e = e - dequantize(q)), "Hardware Acceleration"
// (low-bit codes packed into 32-bit words).
//
// Team geometry: a team of W warps (team_threads = 32 W) owns one bucket; slot s
// of team thread tt covers bucket elements j = (s * team_threads + tt) * 4 ..
// j + 3, so each slot is one coalesced sweep over 128 W consecutive elements.
#pragma once

#include "qc_decode_math.cuh"
#include "qc_device.cuh"
#include "qc_exact_norm.cuh"
#include "qc_internal.h"

namespace qc {

// ------------------------------------------------------------------ statistics

template <int SCHEME>
struct Stats;

template <>
struct Stats<kUniform> {  // min and max of p
    float mn, mx;
    __device__ void init() { mn = __int_as_float(0x7f800000); mx = -mn; }
    __device__ void add(float x) { mn = fminf(mn, x); mx = fmaxf(mx, x); }
    __device__ void warp_reduce() { mn = warp_min(mn); mx = warp_max(mx); }
    __device__ void merge(const Stats &o) { mn = fminf(mn, o.mn); mx = fmaxf(mx, o.mx); }
};

template <>
struct Stats<kTernary> {  // max |p|
    float amax;
    __device__ void init() { amax = 0.0f; }
    __device__ void add(float x) { amax = fmaxf(amax, fabsf(x)); }
    __device__ void warp_reduce() { amax = warp_max(amax); }
    __device__ void merge(const Stats &o) { amax = fmaxf(amax, o.amax); }
};

template <>
struct Stats<kSign> {  // sum of |p| as a double word
    DWord sum;
    __device__ void init() { sum = DWord{0.0f, 0.0f}; }
    __device__ void add(float x) { sum = dw_add(sum, fabsf(x)); }
    __device__ void warp_reduce() { sum = warp_sum(sum); }
    __device__ void merge(const Stats &o) { sum = dw_add(sum, o.sum); }
};

// QSGD: the sum of p^2 as a double word.  Each square is split exactly
// (x * x = hi + lo with lo = fma(x, x, -hi)) and added with an exact TwoSum on
// the high words; the low words are summed in binary32.  A lane sums the
// elements of one window (at most 16) into a fresh double word and merges it
// into its running total; every merge (window, butterfly level, warp) is
// followed by an exact renormalisation so that |lo| <= 2^-24 hi.  With u = 2^-24
// the error of the total is then at most u^2 S (4 * 16^2 + 3 (windows + 12)):
// the 32 low-word roundings of a window of 16 elements err by at most
// 2 * 16 u^2 of its sum each, a renormalised merge by 3 u^2 of the merged sum
// (Finish<kQsgd> uses this bound).
__device__ __forceinline__ DWord dw_renorm(DWord a) {
    const float s = __fadd_rn(a.hi, a.lo);  // |lo| <= hi: Fast2Sum is exact
    return DWord{s, __fsub_rn(a.lo, __fsub_rn(s, a.hi))};
}

template <>
struct Stats<kQsgd> {
    DWord sum;
    __device__ void init() { sum = DWord{0.0f, 0.0f}; }
    __device__ void add(float x) {
        const float hi = __fmul_rn(x, x);
        sum = dw_add(sum, DWord{hi, __fmaf_rn(x, x, -hi)});
    }
    __device__ void warp_reduce() {
        sum = dw_renorm(sum);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            DWord p{__shfl_xor_sync(kFull, sum.hi, o), __shfl_xor_sync(kFull, sum.lo, o)};
            sum = dw_renorm(dw_add(sum, p));
        }
    }
    __device__ void merge(const Stats &o) { sum = dw_renorm(dw_add(sum, o.sum)); }
};

// Per-bucket quantization parameters derived from the statistics.
struct BucketParams {
    float a;           // UNIFORM: min (offset); SIGN / TERNARY: s; QSGD: unit
    float scale;       // UNIFORM: (max - min) / L
    float hi = 0.0f;   // CLIP: the upper bound elements are clamped to
    bool exact = false;  // QSGD: the norm needs the exact path (qc_exact_norm.cuh)
};

template <int SCHEME, int BITS>
struct Finish;

template <int BITS>
struct Finish<kUniform, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kUniform> &st, uint32_t) {
        const float mn = positive_zero(st.mn), mx = positive_zero(st.mx);
        constexpr float L = static_cast<float>((1u << BITS) - 1u);
        return BucketParams{mn, __fdiv_rn(__fsub_rn(mx, mn), L)};
    }
};

template <int BITS>
struct Finish<kTernary, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kTernary> &st, uint32_t) {
        return BucketParams{positive_zero(st.amax), 0.0f};
    }
};

template <int BITS>
struct Finish<kSign, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kSign> &st, uint32_t cnt) {
        return BucketParams{dw_div(st.sum, static_cast<float>(cnt)), 0.0f};
    }
};

// QSGD: unit = nrm / s with s = 2^(BITS-1) - 1, where nrm is the binary32
// rounding of sqrt(S), S the exact sum of squares.  From the renormalised
// double word (hi, lo) ~ S: r0 = sqrt(hi) correctly rounded, the remainder
// hi - r0^2 is exact by fma, and (remainder + lo) / (2 r0) is the first-order
// correction, so N = r0 + corr is sqrt(S) within a relative
//   half the sum's bound + 4.2 u^2     (u = 2^-24; the remainder, the two
// roundings and the second-order term of the square root).  nrm = fl(N), and
// `exact` is set when N lies within twice that bound (plus the 2^-46 that the
// evaluation of its distance may err) of a midpoint between nrm and a
// neighbour, or when hi lies outside [2^-60, 2^124] (squares whose low words
// are not exact, or sums near overflow): such buckets take the exact path.
template <int BITS>
__device__ __forceinline__ BucketParams qsgd_params(float nrm) {
    constexpr float kS = static_cast<float>((1u << (BITS - 1)) - 1u);
    const float unit = __fdiv_rn(nrm, kS);
    return BucketParams{unit, unit};
}

template <int BITS>
struct Finish<kQsgd, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kQsgd> &st, uint32_t cnt) {
        const float hi = st.sum.hi;
        // hi == 0 (a zero bucket, or squares below the binary32 range) goes the exact way too
        if (!(hi >= 0x1p-60f && hi <= 0x1p124f)) {
            BucketParams bp = qsgd_params<BITS>(0.0f);
            bp.exact = true;
            return bp;
        }
        const float r0 = __fsqrt_rn(hi);
        const float rem = __fadd_rn(__fmaf_rn(-r0, r0, hi), st.sum.lo);
        const float corr = __fdiv_rn(rem, __fmul_rn(2.0f, r0));
        const float nrm = __fadd_rn(r0, corr);
        // N - nrm, to within 2^-47 nrm (r0 - nrm is exact: they are within a few ulps)
        const float d = __fadd_rn(__fsub_rn(r0, nrm), corr);
        const uint32_t nb = __float_as_uint(nrm);
        const float half_ulp = __uint_as_float((nb & 0x7F800000u) - (24u << 23));  // nrm >= 2^-30: normal
        const bool pow2 = (nb & 0x7FFFFFu) == 0u;
        const float windows = static_cast<float>((cnt + 511u) / 512u);
        // twice the bound on |N - sqrt(S)| / nrm, plus the evaluation slack
        const float rel = __fmaf_rn(3.0f * 0x1p-48f, windows, (1024.0f + 36.0f + 8.4f) * 0x1p-48f) +
                          0x1p-46f;
        const float slack = __fmul_rn(rel, nrm);
        const bool near_up = d >= __fsub_rn(half_ulp, slack);
        const bool near_dn = -d >= __fsub_rn(pow2 ? __fmul_rn(half_ulp, 0.5f) : half_ulp, slack);
        BucketParams bp = qsgd_params<BITS>(nrm);
        bp.exact = near_up || near_dn;
        return bp;
    }
};

template <>
struct Stats<kLog> : Stats<kTernary> {};  // max |p|

template <int BITS>
struct Finish<kLog, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kLog> &st, uint32_t) {
        return BucketParams{positive_zero(st.amax), 0.0f};
    }
};

// CLIP: the bounds are order statistics found by team_percentiles(), not a
// running reduction, so the add/merge operations are never used.
template <>
struct Stats<kClip> {
    float mn, mx;
    __device__ void init() { mn = mx = 0.0f; }
    __device__ void add(float) {}
    __device__ void warp_reduce() {}
    __device__ void merge(const Stats &) {}
};

template <int BITS>
struct Finish<kClip, BITS> {
    static __device__ __forceinline__ BucketParams run(const Stats<kClip> &st, uint32_t) {
        constexpr float L = static_cast<float>((1u << BITS) - 1u);
        const float mn = positive_zero(st.mn), mx = positive_zero(st.mx);
        return BucketParams{mn, __fdiv_rn(__fsub_rn(mx, mn), L), mx};
    }
};

// ------------------------------------------------------------- per element

// Code and dequantized value of one element.
template <int SCHEME, int BITS, bool SR>
__device__ __forceinline__ uint32_t quantize(float p, float u, const BucketParams &bp,
                                             float &deq) {
    if constexpr (SCHEME == kUniform || SCHEME == kClip) {
        if constexpr (SCHEME == kClip) p = fminf(fmaxf(p, bp.a), bp.hi);  // clamp into [mn, mx]
        constexpr uint32_t L = (1u << BITS) - 1u;
        if (bp.scale == 0.0f) {
            deq = bp.a;
            return 0u;
        }
        const float t = __fdiv_rn(__fsub_rn(p, bp.a), bp.scale);
        uint32_t q = rint_small(t);
        if constexpr (SR) {
            // floor(t) = rint(t) - [rint(t) > t]; frac = t - floor(t) is exact
            if (small_uint_to_float(q) > t) q -= 1u;
            const float fr = __fsub_rn(t, small_uint_to_float(q));
            q += (u < fr) ? 1u : 0u;
        }
        q = min(q, L);
        deq = __fmaf_rn(small_uint_to_float(q), bp.scale, bp.a);
        return q;
    } else if constexpr (SCHEME == kQsgd) {
        // the uniform level of |p| with min 0 and scale = unit, under a sign bit
        constexpr uint32_t S = (1u << (BITS - 1)) - 1u;
        const uint32_t neg = p < 0.0f ? 1u : 0u;
        const float unit = bp.a;
        uint32_t q = 0u;
        if (unit != 0.0f) {
            const float t = __fdiv_rn(fabsf(p), unit);
            q = rint_small(t);
            if constexpr (SR) {
                if (small_uint_to_float(q) > t) q -= 1u;
                const float fr = __fsub_rn(t, small_uint_to_float(q));
                q += (u < fr) ? 1u : 0u;
            }
            q = min(q, S);
        }
        const float mag = __fmul_rn(small_uint_to_float(q), unit);
        deq = neg ? -mag : mag;
        return (neg << (BITS - 1)) | q;
    } else if constexpr (SCHEME == kLog) {
        // levels 0 and s * 2^(j - J): x = |p| / s sits between two levels; its
        // exponent gives the lower one and its mantissa the position between
        constexpr int J = (1 << (BITS - 1)) - 1;
        const uint32_t neg = p < 0.0f ? 1u : 0u;
        const float s = bp.a;
        uint32_t lvl = 0u;
        if (s != 0.0f) {
            const float x = __fdiv_rn(fabsf(p), s);
            const uint32_t xb = __float_as_uint(x);
            const int e = static_cast<int>(xb >> 23) - 127;  // x is normal here when e >= 1 - J
            if (x >= 1.0f) {
                lvl = J;
            } else if (e >= 1 - J) {
                const uint32_t j0 = static_cast<uint32_t>(e + J);
                const float m = __fsub_rn(__uint_as_float((xb & 0x7FFFFFu) | 0x3F800000u), 1.0f);
                bool up;
                if constexpr (SR) up = u < m;
                else up = m > 0.5f || (m == 0.5f && (j0 & 1u));
                lvl = (j0 + (up ? 1u : 0u)) & static_cast<uint32_t>(J);  // a non-finite x stays in its field
            } else {
                // below the smallest level 2^(1-J): the position x / 2^(1-J), exact
                const float f = __fmul_rn(x, __uint_as_float(static_cast<uint32_t>(127 + J - 1) << 23));
                bool up;
                if constexpr (SR) up = u < f;
                else up = f > 0.5f;
                lvl = up ? 1u : 0u;
            }
        }
        const float mag = lvl ? __fmul_rn(s, __uint_as_float((lvl + 127u - J) << 23)) : 0.0f;
        deq = neg ? -mag : mag;
        return (neg << (BITS - 1)) | lvl;
    } else if constexpr (SCHEME == kSign) {
        const bool pos = p >= 0.0f;
        deq = pos ? bp.a : -bp.a;
        return pos ? 1u : 0u;
    } else {  // ternary
        const float s = bp.a;
        if (s == 0.0f) {
            deq = 0.0f;
            return 1u;
        }
        const float pr = __fdiv_rn(fabsf(p), s);
        const bool keep = SR ? (u < pr) : (pr > 0.5f);
        if (!keep) {
            deq = 0.0f;
            return 1u;
        }
        deq = p > 0.0f ? s : -s;
        return p > 0.0f ? 2u : 0u;
    }
}

// ------------------------------------------------- division-free decisions
//
// The divisions t = (p - mn) / scale (uniform) and pr = |p| / s (ternary) only
// decide an integer: a level, a floor, or a comparison with a draw u.  With
// rinv = RN(1 / scale) the product ta = RN(d * rinv) is within
// 3 * 2^-24 * (d / scale) of d / scale, hence within
//   delta = (L + 1) * 2^-22        (uniform; d / scale <= L (1 + 2^-22))
//   delta = 2^-22                  (ternary; |p| / s <= 1)
// of the correctly rounded quotient t = RN(d / scale).  When ta is farther than
// 2 * delta from every decision boundary (half-integers for nearest rounding;
// integers and u for stochastic rounding; u or 1/2 for ternary) the decision
// taken on ta is the decision on t, so the code is the one the IEEE division
// gives.  Otherwise the element is recomputed with the division.  The bound
// needs rinv to be a normal number: buckets whose scale lies outside
// [2^-125, 2^125] (including scale == 0) use the division throughout.
struct FastQ {
    float rinv;
    float delta2;  // twice the bound, covering the rounding of u - ta as well
    bool usable;
};

template <int SCHEME, int BITS>
__device__ __forceinline__ FastQ fast_params(const BucketParams &bp) {
    const float d = (SCHEME == kUniform || SCHEME == kClip) ? bp.scale : bp.a;
    FastQ f;
    const bool normal = d >= 0x1p-125f && d <= 0x1p125f;
    f.usable = SCHEME == kSign || normal;  // the sign code needs no division
    f.rinv = (SCHEME != kSign && normal) ? __frcp_rn(d) : 0.0f;
    f.delta2 = (SCHEME == kUniform || SCHEME == kClip) ? static_cast<float>(1u << BITS) * 0x1p-21f
               : SCHEME == kQsgd     ? static_cast<float>(1u << (BITS - 1)) * 0x1p-21f
               : SCHEME == kLog      ? 0x1p-20f
                                     : 0x1p-21f;
    return f;
}

// Logarithmic level index from xa = fl(|p| * rinv) instead of x = fl(|p| / s).
// |xa - x| < 1.5 * 2^-23 * x, so the position between two levels (the mantissa
// fraction m of x, or f = x * 2^(J-1) below the smallest level; an absolute
// error under 2^-22 + 2^-24 there, subnormal quotients included) moves by less
// than 2^-21.  The decision taken on xa is the decision on x unless the
// position lies within delta2 = 2^-20 of a decision boundary -- 1/2 for nearest
// rounding, u for stochastic rounding -- or, for stochastic rounding, of the
// edge of its binade, where x and xa may sit in neighbouring binades and the
// position jumps from 1 to 0 (for nearest rounding both sides of that jump give
// the same level).  Those elements set redo.  |p| == s is the top level exactly;
// any other |p| has x < 1.  Both positions are formed and one is selected, so
// the element takes no branch; the edge test also flags positions below delta2
// under the smallest level, which only sends a few more elements to the
// division.
template <int BITS, bool SR>
__device__ __forceinline__ uint32_t log_level_fast(float ap, float s, float u, const FastQ &fq,
                                                   bool &redo) {
    constexpr int J = (1 << (BITS - 1)) - 1;
    const float xa = __fmul_rn(ap, fq.rinv);
    const uint32_t xb = __float_as_uint(xa);
    const bool binade = xb >= (static_cast<uint32_t>(128 - J) << 23);  // e >= 1 - J
    const float pos = binade ? __fsub_rn(__uint_as_float((xb & 0x7FFFFFu) | 0x3F800000u), 1.0f)
                             : __fmul_rn(xa, __uint_as_float(static_cast<uint32_t>(127 + J - 1) << 23));
    const uint32_t j0 = binade ? (xb >> 23) - static_cast<uint32_t>(127 - J) : 0u;
    bool up;
    if constexpr (SR) {
        up = u < pos;
        redo = (fabsf(__fsub_rn(u, pos)) <= fq.delta2) |
               (fabsf(__fsub_rn(pos, 0.5f)) >= 0.5f - fq.delta2) | (xa >= 1.0f);
    } else {
        up = pos > 0.5f;  // a tie is within delta2 and recomputed
        redo = (fabsf(__fsub_rn(pos, 0.5f)) <= fq.delta2) | (xa >= 1.0f);
    }
    const bool top = ap == s;
    redo = redo && !top;
    return top ? static_cast<uint32_t>(J) : j0 + (up ? 1u : 0u);
}

// Code and dequantized value of one element from ta; sets redo when the
// decision is within reach of the approximation error.
template <int SCHEME, int BITS, bool SR>
__device__ __forceinline__ uint32_t quantize_fast(float p, float u, const BucketParams &bp,
                                                  const FastQ &fq, float &deq, bool &redo) {
    if constexpr (SCHEME == kUniform || SCHEME == kClip) {
        if constexpr (SCHEME == kClip) p = fminf(fmaxf(p, bp.a), bp.hi);
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
        const float ta = __fmul_rn(__fsub_rn(p, bp.a), fq.rinv);
        float qf;
        uint32_t q;
        if constexpr (!SR) {
            const float y = __fadd_rn(ta, kMagic);  // rint(ta) in the low mantissa bits
            q = __float_as_uint(y) - 0x4B400000u;
            qf = __fsub_rn(y, kMagic);
            redo = fabsf(__fsub_rn(ta, qf)) >= 0.5f - fq.delta2;
        } else {
            // floor(t) + [u < t - floor(t)] = ceil(t - u): one decision instead
            // of two.  x = fl(ta - u) is within delta2 of t - u (ta's bound and
            // the subtraction's rounding, (L + 1) 2^-24 at most), so ceil(x) is
            // the level unless x lies within delta2 of an integer (then the exact
            // path decides).  x > -1, and rint(x) = -1 wraps to 0 with the +1.
            const float x = __fsub_rn(ta, u);
            const float y = __fadd_rn(x, kMagic);  // rint(x) in the low mantissa bits
            const float rf = __fsub_rn(y, kMagic);
            const float dx = __fsub_rn(x, rf);     // exact
            const bool up = dx > 0.0f;             // ceil(x) = rint(x) + [x > rint(x)]
            q = __float_as_uint(y) - 0x4B400000u + (up ? 1u : 0u);
            qf = up ? __fadd_rn(rf, 1.0f) : rf;
            redo = fabsf(dx) <= fq.delta2;
        }
        // no clamp: 0 <= ta <= L (1 + 2^-22), so a level above L needs ta within
        // reach of L + 1/2 (impossible) or of the integer L (flagged by redo).
        // The mask keeps a non-finite element's code inside its own field.
        deq = __fmaf_rn(qf, bp.scale, bp.a);
        return q & ((1u << BITS) - 1u);
    } else if constexpr (SCHEME == kQsgd) {
        constexpr float kMagic = 12582912.0f;
        const uint32_t neg = p < 0.0f ? 1u : 0u;
        const float ta = __fmul_rn(fabsf(p), fq.rinv);
        float qf;
        uint32_t q;
        if constexpr (!SR) {
            const float y = __fadd_rn(ta, kMagic);
            q = __float_as_uint(y) - 0x4B400000u;
            qf = __fsub_rn(y, kMagic);
            redo = fabsf(__fsub_rn(ta, qf)) >= 0.5f - fq.delta2;
        } else {  // ceil(ta - u), as for the uniform levels
            const float x = __fsub_rn(ta, u);
            const float y = __fadd_rn(x, kMagic);
            const float rf = __fsub_rn(y, kMagic);
            const float dx = __fsub_rn(x, rf);
            const bool up = dx > 0.0f;
            q = __float_as_uint(y) - 0x4B400000u + (up ? 1u : 0u);
            qf = up ? __fadd_rn(rf, 1.0f) : rf;
            redo = fabsf(dx) <= fq.delta2;
        }
        // no clamp: t <= S (1 + 2^-22); a level above S would be flagged by redo
        // (the mask keeps a non-finite element's code inside its own field)
        const float mag = __fmul_rn(qf, bp.a);
        deq = neg ? -mag : mag;
        return (neg << (BITS - 1)) | (q & ((1u << (BITS - 1)) - 1u));
    } else if constexpr (SCHEME == kTernary) {
        const float s = bp.a;
        const float pa = __fmul_rn(fabsf(p), fq.rinv);
        bool keep;
        if constexpr (SR) {
            keep = u < pa;
            redo = fabsf(__fsub_rn(u, pa)) <= fq.delta2;
        } else {
            keep = pa > 0.5f;
            redo = fabsf(__fsub_rn(pa, 0.5f)) <= fq.delta2;
        }
        if (!keep) {
            deq = 0.0f;
            return 1u;
        }
        deq = p > 0.0f ? s : -s;
        return p > 0.0f ? 2u : 0u;
    } else if constexpr (SCHEME == kLog) {
        constexpr uint32_t J = (1u << (BITS - 1)) - 1u;
        const uint32_t neg = p < 0.0f ? 1u : 0u;
        const uint32_t lvl = log_level_fast<BITS, SR>(fabsf(p), bp.a, u, fq, redo) & J;
        const float mag = lvl ? __fmul_rn(bp.a, __uint_as_float((lvl + 127u - J) << 23)) : 0.0f;
        deq = neg ? -mag : mag;
        return (neg << (BITS - 1)) | lvl;
    } else {
        redo = false;
        return quantize<SCHEME, BITS, SR>(p, u, bp, deq);
    }
}

// Code of one element from ta; sets redo when the decision is within reach of
// the approximation error (the caller then recomputes it with the division).
template <int SCHEME, int BITS, bool SR>
__device__ __forceinline__ uint32_t code_fast(float p, float u, const BucketParams &bp,
                                              const FastQ &fq, bool &redo) {
    if constexpr (SCHEME == kUniform || SCHEME == kClip) {
        if constexpr (SCHEME == kClip) p = fminf(fmaxf(p, bp.a), bp.hi);
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
        const float ta = __fmul_rn(__fsub_rn(p, bp.a), fq.rinv);
        uint32_t q;
        if constexpr (!SR) {
            const float y = __fadd_rn(ta, kMagic);  // rint(ta) in the low mantissa bits
            q = __float_as_uint(y) - 0x4B400000u;
            redo = fabsf(__fsub_rn(ta, __fsub_rn(y, kMagic))) >= 0.5f - fq.delta2;
        } else {  // ceil(ta - u) (see quantize_fast)
            const float x = __fsub_rn(ta, u);
            const float y = __fadd_rn(x, kMagic);
            const float dx = __fsub_rn(x, __fsub_rn(y, kMagic));
            redo = fabsf(dx) <= fq.delta2;
            q = __float_as_uint(y) - 0x4B400000u + (dx > 0.0f ? 1u : 0u);
        }
        return q & ((1u << BITS) - 1u);  // no clamp needed outside redo (see quantize_fast)
    } else if constexpr (SCHEME == kTernary) {
        const float pa = __fmul_rn(fabsf(p), fq.rinv);
        bool keep;
        if constexpr (SR) {
            const float d = __fsub_rn(u, pa);
            keep = d < 0.0f;
            redo = fabsf(d) <= fq.delta2;
        } else {
            keep = pa > 0.5f;
            redo = fabsf(__fsub_rn(pa, 0.5f)) <= fq.delta2;
        }
        // keep ? (p > 0 ? 2 : 0) : 1; a kept element is never zero
        return keep ? ((__float_as_uint(p) >> 31) ? 0u : 2u) : 1u;
    } else if constexpr (SCHEME == kQsgd) {
        constexpr float kMagic = 12582912.0f;
        const float ta = __fmul_rn(fabsf(p), fq.rinv);
        uint32_t q;
        if constexpr (!SR) {
            const float y = __fadd_rn(ta, kMagic);
            q = __float_as_uint(y) - 0x4B400000u;
            redo = fabsf(__fsub_rn(ta, __fsub_rn(y, kMagic))) >= 0.5f - fq.delta2;
        } else {  // ceil(ta - u)
            const float x = __fsub_rn(ta, u);
            const float y = __fadd_rn(x, kMagic);
            const float dx = __fsub_rn(x, __fsub_rn(y, kMagic));
            redo = fabsf(dx) <= fq.delta2;
            q = __float_as_uint(y) - 0x4B400000u + (dx > 0.0f ? 1u : 0u);
        }
        return ((p < 0.0f ? 1u : 0u) << (BITS - 1)) | (q & ((1u << (BITS - 1)) - 1u));  // no clamp outside redo
    } else if constexpr (SCHEME == kLog) {
        return ((p < 0.0f ? 1u : 0u) << (BITS - 1)) |
               (log_level_fast<BITS, SR>(fabsf(p), bp.a, u, fq, redo) & ((1u << (BITS - 1)) - 1u));
    } else {
        static_assert(SCHEME == kSign, "code_fast: every other scheme has its own branch");
        redo = false;
        return p >= 0.0f ? 1u : 0u;
    }
}

// Exact code of one element (the IEEE division path).
template <int SCHEME, int BITS, bool SR>
__device__ __forceinline__ uint32_t code_exact(float p, float u, const BucketParams &bp) {
    float deq;
    return quantize<SCHEME, BITS, SR>(p, u, bp, deq);
}

// Dequantized value of code c of a packed field, identical to the encoder's deq.
template <int SCHEME, int BITS>
__device__ __forceinline__ float deq_of(uint32_t field, int c, const BucketParams &bp) {
    if constexpr (SCHEME == kUniform || SCHEME == kClip)
        return dequant_code<kUniform, BITS>(field, c, bp.scale, bp.a);
    else return dequant_code<SCHEME, BITS>(field, c, bp.a, bp.a);
}

// ------------------------------------------------------------- slot level

// Adds the valid elements of the lane's slots to the statistics.  FULL: the
// caller guarantees cnt == team_threads * kSlots * 4 (every slot valid), which
// removes the per-slot bounds checks.
template <int SCHEME, bool FULL = false>
__device__ __forceinline__ void accumulate_slots(Stats<SCHEME> &st, const float4 (&p)[kSlots],
                                                 int tt, int team_threads, uint32_t cnt) {
    // QSGD sums a window into a fresh double word and merges it (see Stats<kQsgd>)
    Stats<SCHEME> part;
    if constexpr (SCHEME == kQsgd) part.init();
    Stats<SCHEME> &acc = (SCHEME == kQsgd) ? part : st;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u;
        if (FULL || j + 4u <= cnt) {
            acc.add(p[s].x);
            acc.add(p[s].y);
            acc.add(p[s].z);
            acc.add(p[s].w);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (j + c < cnt) acc.add(get(p[s], c));
        }
    }
    if constexpr (SCHEME == kQsgd) st.merge(part);
}

// The exact sum of the squares of the lane's valid elements (the QSGD norm's
// exact path).
__device__ __forceinline__ void wide_add_slots(WideSum &acc, const float4 (&p)[kSlots], int tt,
                                               int team_threads, uint32_t cnt) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u + c;
            if (j < cnt) wide_add_square(acc, get(p[s], c));
        }
    }
}

// Barrier over one team on named barrier BAR0 + team (the warp itself for W = 1).
template <int BAR0>
__device__ __forceinline__ void team_bar(int W, int team) {
    if (W == 1) {
        __syncwarp();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(BAR0 + team), "r"(W * 32) : "memory");
    }
}

// The exactly rounded norm from every team thread's exact partial sum: a warp
// butterfly, then (W > 1) the warps' sums two limbs at a time through the
// team's slots of the statistics buffer (alternating between its two halves),
// one team barrier per round.  Every thread of the team calls this together
// (the caller's decision is uniform across the team) and gets the same value.
template <int SCHEME, int BAR0>
__device__ __forceinline__ float team_exact_norm(WideSum &acc, Stats<SCHEME> (*red)[kBlock / 32],
                                              int W, int warp, int lane, int team) {
    static_assert(sizeof(Stats<SCHEME>) >= 8, "two limbs per warp slot");
    wide_warp_sum(acc);
    if (W > 1) {
        uint64_t tot[kWideLimbs];
#pragma unroll
        for (int i = 0; i < kWideLimbs; ++i) tot[i] = 0u;
        team_bar<BAR0>(W, team);  // every warp is done with the statistics buffer
        for (int r = 0; r < kWideLimbs; r += 2) {
            uint32_t *mine = reinterpret_cast<uint32_t *>(&red[(r >> 1) & 1][warp]);
            if (lane == 0) {
                mine[0] = acc.w[r];
                mine[1] = acc.w[r + 1];
            }
            team_bar<BAR0>(W, team);
            for (int w = 0; w < W; ++w) {
                const uint32_t *o = reinterpret_cast<const uint32_t *>(&red[(r >> 1) & 1][team * W + w]);
                tot[r] += o[0];
                tot[r + 1] += o[1];
            }
        }
        team_bar<BAR0>(W, team);  // every warp has read the last round
        uint64_t carry = 0;
        for (int i = 0; i < kWideLimbs; ++i) {
            const uint64_t t = tot[i] + carry;
            acc.w[i] = static_cast<uint32_t>(t);
            carry = t >> 32;
        }
    }
    return wide_sqrt_f32(acc);
}

// Quantizes the lane's slots of bucket [b0, b0 + cnt), packs and stores the code
// words, and (with error feedback) stores the new residual.  Element i draws
// with the index draw_base + i (a segment's place in a multi-segment call).  All 32 lanes of the
// warp must call this together (the packing uses shuffles).  FULL as for
// accumulate_slots.
template <int SCHEME, int BITS, bool SR, bool EF, bool FULL = false>
__device__ __forceinline__ void quantize_store_slots(uint32_t *codes, float *err, uint64_t b0,
                                                     uint32_t cnt, int tt, int team_threads,
                                                     int lane, const float4 (&p)[kSlots],
                                                     const BucketParams &bp, uint32_t step,
                                                     const PhiloxKeys &keys, uint64_t draw_base = 0) {
    const FastQ fq = fast_params<SCHEME, BITS>(bp);
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u;
        const uint64_t i = b0 + j;
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (SR) {
            if (FULL || j < cnt) uniform4(draw_base + i, step, keys, u);
        }
        uint32_t field = 0;
        float4 e;
        if ((FULL || j + 4u <= cnt) && fq.usable) {
            float d[4];
            bool redo[4];
            uint32_t q[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                q[c] = quantize_fast<SCHEME, BITS, SR>(get(p[s], c), u[c], bp, fq, d[c], redo[c]);
            if (redo[0] | redo[1] | redo[2] | redo[3]) {  // rare: near a decision boundary
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (redo[c]) q[c] = quantize<SCHEME, BITS, SR>(get(p[s], c), u[c], bp, d[c]);
            }
            field = q[0] | (q[1] << BITS) | (q[2] << (2 * BITS)) | (q[3] << (3 * BITS));
            e = make_float4(__fsub_rn(p[s].x, d[0]), __fsub_rn(p[s].y, d[1]),
                            __fsub_rn(p[s].z, d[2]), __fsub_rn(p[s].w, d[3]));
        } else if (FULL || j + 4u <= cnt) {
            float d0, d1, d2, d3;
            field = quantize<SCHEME, BITS, SR>(p[s].x, u[0], bp, d0) |
                    (quantize<SCHEME, BITS, SR>(p[s].y, u[1], bp, d1) << BITS) |
                    (quantize<SCHEME, BITS, SR>(p[s].z, u[2], bp, d2) << (2 * BITS)) |
                    (quantize<SCHEME, BITS, SR>(p[s].w, u[3], bp, d3) << (3 * BITS));
            e = make_float4(__fsub_rn(p[s].x, d0), __fsub_rn(p[s].y, d1), __fsub_rn(p[s].z, d2),
                            __fsub_rn(p[s].w, d3));
        } else {
            e = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j + c < cnt) {
                    float deq;
                    const float pc = get(p[s], c);
                    field |= quantize<SCHEME, BITS, SR>(pc, u[c], bp, deq) << (c * BITS);
                    set(e, c, __fsub_rn(pc, deq));
                }
            }
        }
        const uint32_t word = gather_word<BITS>(field);
        if ((FULL || j < cnt) && stores_word<BITS>(lane)) __stcs(codes + (i * BITS) / 32u, word);
        if constexpr (EF) {
            if (FULL || j + 4u <= cnt) {
                __stcs(reinterpret_cast<float4 *>(err + i), e);
            } else if (j < cnt) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (j + c < cnt) err[i + c] = get(e, c);
            }
        }
    }
}

template <int SCHEME>
__device__ __forceinline__ void store_meta(float *scale, float *offset, uint64_t k,
                                           const BucketParams &bp) {
    if constexpr (SCHEME == kUniform || SCHEME == kClip) {
        scale[k] = bp.scale;
        offset[k] = bp.a;
    } else {
        scale[k] = bp.a;
    }
}

// Team-wide reduction of the statistics: warp butterflies, then (W > 1) one
// exchange through shared memory.  Every thread of the block (with kNamed, every
// thread of the kBlock consumer threads on named barrier 1) must call it.
template <int SCHEME, bool kNamed = false>
__device__ __forceinline__ void team_reduce(Stats<SCHEME> &st, Stats<SCHEME> (*red)[kBlock / 32],
                                            int &buf, int W, int warp, int lane, int team) {
    st.warp_reduce();
    if (W > 1) {
        if (lane == 0) red[buf][warp] = st;
        if constexpr (kNamed) {
            asm volatile("bar.sync 1, %0;" ::"n"(kBlock) : "memory");
        } else {
            __syncthreads();
        }
        st = red[buf][team * W];
        for (int w = 1; w < W; ++w) st.merge(red[buf][team * W + w]);
        buf ^= 1;
    }
}

// team_reduce for the pipelined kernels, which also tells the team whether every
// thread's wait for the stage succeeded (ok): the warp's vote when a team is one
// warp, else the block barrier that the exchange needs anyway (then block-wide).
template <int SCHEME>
__device__ __forceinline__ bool team_reduce_ok(Stats<SCHEME> &st, Stats<SCHEME> (*red)[kBlock / 32],
                                               int &buf, int W, int warp, int lane, int team,
                                               bool ok) {
    st.warp_reduce();
    if (W > 1) {
        if (lane == 0) red[buf][warp] = st;
        ok = __syncthreads_and(ok) != 0;
        st = red[buf][team * W];
        for (int w = 1; w < W; ++w) st.merge(red[buf][team * W + w]);
        buf ^= 1;
        return ok;
    }
    return __all_sync(kFull, ok);
}

// Team-wide reduction like team_reduce, synchronised only within the team
// (team_sync), so teams proceed independently.  Every thread of the team calls
// it together.
template <int SCHEME>
__device__ __forceinline__ void team_reduce_local(Stats<SCHEME> &st, Stats<SCHEME> (*red)[kBlock / 32],
                                                  int &buf, int W, int warp, int lane, int team);

// The exact norm of a bucket whose elements the team holds in its slots (one
// window).  Inlined like the rest of the exact path: a call would make the
// kernel keep its live registers in the call convention's registers, costing
// the main loop occupancy, while the inlined path keeps its limbs on the stack.
template <int SCHEME, int BAR0>
__device__ __forceinline__ float team_exact_norm_slots(const float4 (&p)[kSlots], int tt,
                                                    int team_threads, uint32_t cnt,
                                                    Stats<SCHEME> (*red)[kBlock / 32], int W,
                                                    int warp, int lane, int team) {
    WideSum acc;
    wide_zero(acc);
    wide_add_slots(acc, p, tt, team_threads, cnt);
    return team_exact_norm<SCHEME, BAR0>(acc, red, W, warp, lane, team);
}

// ------------------------------------------------------------- percentiles

// Unsigned keys that order like the floats (-0 just below +0).
__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// 256-bin histograms with 16-bit counters, two bins per word (a bucket holds at
// most 4096 elements, so a count never carries into its neighbour).
constexpr int kHistWords = 128;
constexpr int kHistTeamWords = 3 * 2 * kHistWords;  // 3 rotating buffers x (low, high)

__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin) {
    atomicAdd(h + (bin >> 1), 1u << ((bin & 1u) << 4));
}

// The bin of a histogram of 64 * WPL bins (WPL packed words per lane) that
// holds rank r (0-based); r becomes the rank within that bin.  Every lane of
// the calling warp gets the same answer.
template <int WPL>
__device__ __forceinline__ uint32_t hist_find(const uint32_t *h, uint32_t &r, int lane) {
    uint32_t w[WPL], sum = 0u;
#pragma unroll
    for (int q = 0; q < WPL; ++q) {
        w[q] = h[WPL * lane + q];
        sum += (w[q] & 0xFFFFu) + (w[q] >> 16);
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - sum;
    const bool mine = excl <= r && r < incl;
    const int owner = __ffs(__ballot_sync(kFull, mine)) - 1;
    uint32_t bin = 0u, before = 0u, acc = excl;
    bool found = false;
#pragma unroll
    for (int k = 0; k < 2 * WPL; ++k) {
        const uint32_t c = (k & 1) ? (w[k >> 1] >> 16) : (w[k >> 1] & 0xFFFFu);
        if (!found && r < acc + c) {
            bin = static_cast<uint32_t>(2 * WPL * lane + k);
            before = acc;
            found = true;
        }
        acc += c;
    }
    bin = __shfl_sync(kFull, bin, owner);
    before = __shfl_sync(kFull, before, owner);
    r -= before;
    return bin;
}

// Barrier over one team: the warp itself, or named barrier 1 + team over its W
// warps (teams never wait for one another).
__device__ __forceinline__ void team_sync(int W, int team) {
    if (W == 1) {
        __syncwarp();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(W * 32) : "memory");
    }
}

// Whether v holds on every thread of the team (the team's named barrier).
__device__ __forceinline__ bool team_all(bool v, int W, int team) {
    if (W == 1) return __all_sync(kFull, v);
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(1 + team), "r"(W * 32)
        : "memory");
    return r != 0u;
}

// Full radix selection: the keys of ranks r_lo and r_hi (0-based, ascending)
// among the cnt valid keys of the team's slots, by four rounds of 8-bit
// selection, most significant byte first.
// Round 0 builds one histogram of every element's top byte; later rounds
// count only the elements sharing the bytes already fixed for each rank.  The
// three buffers of `region` (3 x 2 x kHistWords words, all zero on entry)
// rotate: a round fills one, and after the barrier clears the one filled two
// rounds earlier, which every warp has finished reading.  Every thread of the
// team calls this together; `region` is left with arbitrary contents.
__device__ __forceinline__ void team_radix_select(const uint32_t (&keys)[kSlots][4], uint32_t cnt,
                                                  int tt, int team_threads, int W, int team,
                                                  int lane, uint32_t *region, uint32_t r_lo,
                                                  uint32_t r_hi, uint32_t &key_lo, uint32_t &key_hi) {
    uint32_t pre_lo = 0u, pre_hi = 0u;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *h = region + (pass % 3) * (2 * kHistWords);
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u + c;
                if (j < cnt) {
                    const uint32_t key = keys[s][c];
                    const uint32_t d = (key >> shift) & 0xFFu;
                    if (pass == 0) {
                        hist_add(h, d);
                    } else {
                        const uint32_t top = key >> (shift + 8);
                        if (top == (pre_lo >> (shift + 8))) hist_add(h, d);
                        if (top == (pre_hi >> (shift + 8))) hist_add(h + kHistWords, d);
                    }
                }
            }
        }
        team_sync(W, team);
        pre_lo |= hist_find<kHistWords / 32>(h, r_lo, lane) << shift;
        pre_hi |= hist_find<kHistWords / 32>(pass == 0 ? h : h + kHistWords, r_hi, lane) << shift;
        uint32_t *old = region + ((pass + 2) % 3) * (2 * kHistWords);
        for (int i = tt; i < 2 * kHistWords; i += team_threads) old[i] = 0u;
    }
    key_lo = pre_lo;
    key_hi = pre_hi;
}

// The element of rank r (0-based, by key) among the m keys of `list`; every
// lane of the calling warp gets it.  Each lane ranks its own candidates
// against the whole list (broadcast reads), so a value with fewer than r + 1
// keys below it and more than r keys at or below it is the answer.
__device__ __forceinline__ uint32_t list_select(const uint32_t *list, uint32_t m, uint32_t r,
                                                int lane) {
    uint32_t ans = 0u;
    bool found = false;
    for (uint32_t i = static_cast<uint32_t>(lane); i < m; i += 32u) {
        const uint32_t x = list[i];
        uint32_t less = 0u, leq = 0u;
        for (uint32_t j = 0; j < m; ++j) {
            const uint32_t y = list[j];
            less += y < x ? 1u : 0u;
            leq += y <= x ? 1u : 0u;
        }
        if (less <= r && r < leq) {
            ans = x;
            found = true;
        }
    }
    const uint32_t who = __ballot_sync(kFull, found);
    return __shfl_sync(kFull, ans, __ffs(who) - 1);
}

// Layout of a team's selection region (words): two sets (alternating between
// buckets) of three 256-bin histograms (top key byte; second byte for each
// rank); the short lists of keys sharing both bytes; two sets of counters; the
// results; the two candidate lists of bucket / 4 keys each.  The full radix
// selection overlays the two histogram sets with its three rotating buffers.
constexpr int kShortCap = 64;
constexpr int kSelSet = 3 * kHistWords;
static_assert(2 * kSelSet == kHistTeamWords, "the radix buffers overlay the histogram sets");
constexpr int kSelShortLo = 2 * kSelSet, kSelShortHi = kSelShortLo + kShortCap;
constexpr int kSelCount = kSelShortHi + kShortCap;  // 2 sets x (list lo, list hi, short lo, short hi)
constexpr int kSelResult = kSelCount + 8;
constexpr int kSelLists = kSelResult + 4;
static_assert(kSelLists == kSelFixedWords, "sel_region_words() in qc_internal.h");

// The element of rank r among the keys of `list` that have top 16 bits `pre`,
// computed by one warp: the matching keys are gathered into `sub` (ballot
// compaction), then each lane ranks its own against all of them.  Returns
// false if more than kShortCap keys match (the caller falls back).
__device__ __forceinline__ bool list_select16(const uint32_t *list, uint32_t m, uint32_t pre,
                                              uint32_t r, uint32_t *sub, int lane,
                                              uint32_t &out) {
    uint32_t ms = 0u;
    for (uint32_t i0 = 0; i0 < m; i0 += 32u) {
        const uint32_t i = i0 + static_cast<uint32_t>(lane);
        const uint32_t x = i < m ? list[i] : 0u;
        const bool hit = i < m && (x >> 16) == pre;
        const uint32_t mask = __ballot_sync(kFull, hit);
        const uint32_t at = ms + __popc(mask & ((1u << lane) - 1u));
        if (hit && at < kShortCap) sub[at] = x;
        ms += __popc(mask);
    }
    if (ms > kShortCap) return false;
    __syncwarp();
    out = list_select(sub, ms, r, lane);
    return true;
}

template <int SCHEME>
__device__ __forceinline__ void team_reduce_local(Stats<SCHEME> &st, Stats<SCHEME> (*red)[kBlock / 32],
                                                  int &buf, int W, int warp, int lane, int team) {
    st.warp_reduce();
    if (W > 1) {
        if (lane == 0) red[buf][warp] = st;
        team_sync(W, team);
        st = red[buf][team * W];
        for (int w = 1; w < W; ++w) st.merge(red[buf][team * W + w]);
        buf ^= 1;
    }
}

// The keys of ranks r_lo and r_hi (0-based, ascending; NR = 1: r_lo only)
// among the cnt valid keys of the team's slots.  Round 0 histograms every key's
// top byte; every warp finds the bins holding the ranks.  Round 1 histograms
// the second byte of the keys in those bins, one histogram per rank, and
// appends them to a list per rank.  After the barrier one warp per rank finds
// the second byte, gathers the listed keys sharing both bytes (a handful for
// spread-out data) and selects the exact key among them.  Buckets whose bin
// holds more than a quarter of the bucket, or whose two-byte prefix is shared
// by more than kShortCap keys (constant buckets, heavy ties), take the full
// radix selection.  Histograms and counters alternate between two sets
// (`parity`, flipped per call): a set is cleared after the third barrier of
// one bucket and next used, already clear, by the bucket after, so the fast
// path needs three barriers.  cnt > 0; every thread of the team calls this
// together.  FULL: every slot is valid.
template <int NR, bool FULL>
__device__ __forceinline__ void team_select(const uint32_t (&key)[kSlots][4], uint32_t cnt,
                                            uint32_t bucket, uint32_t k_lo, uint32_t k_hi, int tt,
                                            int team_threads, int W, int team, int warp_in_team,
                                            int lane, uint32_t *region, uint32_t &parity,
                                            uint32_t &key_lo, uint32_t &key_hi) {
    const uint32_t cap = bucket / 4u;
    uint32_t *set = region + parity * kSelSet;
    uint32_t *hist0 = set, *hist_lo = set + kHistWords, *hist_hi = set + 2 * kHistWords;
    uint32_t *count = region + kSelCount + 4 * parity;
    uint32_t *list_lo = region + kSelLists, *list_hi = list_lo + cap;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u + c;
            if (FULL || j < cnt) hist_add(hist0, key[s][c] >> 24);
        }
    }
    team_sync(W, team);  // (1)
    uint32_t r_lo = k_lo, r_hi = k_hi;
    const uint32_t b_lo = hist_find<kHistWords / 32>(hist0, r_lo, lane);
    const uint32_t b_hi = NR > 1 ? hist_find<kHistWords / 32>(hist0, r_hi, lane) : 0u;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u + c;
            const uint32_t top = key[s][c] >> 24, d = (key[s][c] >> 16) & 0xFFu;
            if ((FULL || j < cnt) && top == b_lo) {
                hist_add(hist_lo, d);
                const uint32_t at = atomicAdd(count, 1u);
                if (at < cap) list_lo[at] = key[s][c];
            }
            if (NR > 1 && (FULL || j < cnt) && top == b_hi) {
                hist_add(hist_hi, d);
                const uint32_t at = atomicAdd(count + 1, 1u);
                if (at < cap) list_hi[at] = key[s][c];
            }
        }
    }
    team_sync(W, team);  // (2)
    const uint32_t m_lo = count[0], m_hi = count[1];
    bool fast = m_lo <= cap && m_hi <= cap;
    key_lo = key_hi = 0u;
    if (fast) {
        // the selecting warps flag an overflowing short list in the counters
        if (warp_in_team == 0) {
            const uint32_t pre = (b_lo << 8) | hist_find<kHistWords / 32>(hist_lo, r_lo, lane);
            uint32_t x = 0u;
            const bool ok = list_select16(list_lo, m_lo, pre, r_lo, region + kSelShortLo, lane, x);
            if (lane == 0) {
                region[kSelResult] = x;
                count[2] = ok ? 0u : 1u;
            }
        }
        if (NR > 1 && warp_in_team == (W > 1 ? 1 : 0)) {
            const uint32_t pre = (b_hi << 8) | hist_find<kHistWords / 32>(hist_hi, r_hi, lane);
            uint32_t x = 0u;
            const bool ok = list_select16(list_hi, m_hi, pre, r_hi, region + kSelShortHi, lane, x);
            if (lane == 0) {
                region[kSelResult + 1] = x;
                count[3] = ok ? 0u : 1u;
            }
        }
        team_sync(W, team);  // (3)
        fast = count[2] == 0u && count[3] == 0u;
        key_lo = region[kSelResult];
        key_hi = region[kSelResult + 1];
    }
    if (fast) {
        // this set is next used two buckets from now; the other set and its
        // counters were cleared during the previous bucket
        for (int i = tt; i < kSelSet; i += team_threads) set[i] = 0u;
        if (tt == 0) {
            uint32_t *other = region + kSelCount + 4 * (parity ^ 1u);
            other[0] = other[1] = other[2] = other[3] = 0u;
        }
    } else {
        team_sync(W, team);  // every thread has read the counters
        for (int i = tt; i < 2 * kSelSet; i += team_threads) region[i] = 0u;
        team_sync(W, team);
        team_radix_select(key, cnt, tt, team_threads, W, team, lane, region, k_lo,
                          NR > 1 ? k_hi : k_lo, key_lo, key_hi);
        team_sync(W, team);  // every warp is done with the last round's buffer
        for (int i = tt; i < 2 * kSelSet; i += team_threads) region[i] = 0u;
        for (int i = tt; i < 8; i += team_threads) region[kSelCount + i] = 0u;
        team_sync(W, team);  // all clear before the next bucket
    }
    parity ^= 1u;
}

// The nearest-rank 1st and 99th percentiles of the cnt valid elements in the
// team's slots: the order keys of ranks ceil(cnt/100) - 1 and
// ceil(99 cnt/100) - 1 (0-based), by team_select.
template <bool FULL>
__device__ __forceinline__ void team_percentiles(const float4 (&p)[kSlots], uint32_t cnt, uint32_t bucket,
                                                 int tt, int team_threads, int W, int team,
                                                 int warp_in_team, int lane, uint32_t *region,
                                                 uint32_t &parity, float &lo, float &hi) {
    uint32_t key[kSlots][4];
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
#pragma unroll
        for (int c = 0; c < 4; ++c) key[s][c] = order_key(get(p[s], c));
    uint32_t key_lo, key_hi;
    team_select<2, FULL>(key, cnt, bucket, (cnt + 99u) / 100u - 1u, (99u * cnt + 99u) / 100u - 1u,
                         tt, team_threads, W, team, warp_in_team, lane, region, parity, key_lo,
                         key_hi);
    lo = key_value(key_lo);
    hi = key_value(key_hi);
}

}  // namespace qc
