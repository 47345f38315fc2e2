// qc_encode.cu -- sender half of the codec: error-feedback quantization of a
// flat gradient, one single-pass kernel per (scheme, bits, rounding, dtype, EF).
//
// "Quantization for Communication", sections "Quantization Schemes" (uniform
// min/max levels, stochastic rounding), "Quantized SGD Algorithms" (TernGrad,
// SignSGD), "Error Feedback for Quantization" (e = e + g; q = Q(e);
// e = e - deq(q)), "Hardware Acceleration" (packed low-bit words).
//
// Layout of the work: a team of W warps owns one bucket.  Each lane holds 4
// float4 slots; slot s of team thread t covers bucket elements
// (s * 32W + t) * 4 .. +3, so every slot is one fully coalesced 512W-byte
// (fp32) sweep.  A bucket of up to 512W elements stays in registers between
// the statistics pass and the quantize pass (one HBM read, one write); larger
// buckets take the statistics pass and then re-read the bucket, which is still
// resident in L2.  Reductions are warp butterflies plus one shared-memory step
// across the team's warps.
#include "qc_device.cuh"
#include "qc_internal.h"

namespace qc {
namespace {

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

// Per-bucket quantization parameters derived from the statistics.
struct BucketParams {
    float a;  // UNIFORM: min (offset); SIGN / TERNARY: s
    float scale;  // UNIFORM: (max - min) / L
};

template <int SCHEME, int BITS>
struct Finish {
    static __device__ __forceinline__ BucketParams run(const Stats<SCHEME> &st, uint32_t cnt);
};

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

// ------------------------------------------------------------- per element

// Code and dequantized value of one element.
template <int SCHEME, int BITS, bool SR>
__device__ __forceinline__ uint32_t quantize(float p, float u, const BucketParams &bp,
                                             float &deq) {
    if constexpr (SCHEME == kUniform) {
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

// --------------------------------------------------------------- the kernel

template <typename TIn, bool EF>
__device__ __forceinline__ void load_slots(const EncodeParams &P, uint64_t b0, uint32_t cnt,
                                           uint32_t w0, int tt, int team_threads,
                                           float4 (&p)[kSlots], bool (&full)[kSlots]) {
    const TIn *g = static_cast<const TIn *>(P.grad);
    float4 gv[kSlots], ev[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = w0 + static_cast<uint32_t>(s * team_threads + tt) * 4u;
        const uint64_t i = b0 + j;
        full[s] = j + 4u <= cnt;
        gv[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        ev[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (full[s]) {
            gv[s] = GradLoad<TIn>::full(g, i);
            if constexpr (EF) ev[s] = __ldcs(reinterpret_cast<const float4 *>(P.err + i));
        } else if (j < cnt) {  // ragged end of the array: element-wise
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j + c < cnt) {
                    set(gv[s], c, GradLoad<TIn>::one(g, i + c));
                    if constexpr (EF) set(ev[s], c, __ldcs(P.err + i + c));
                }
            }
        }
    }
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        if constexpr (EF) {
            p[s] = make_float4(__fadd_rn(ev[s].x, gv[s].x), __fadd_rn(ev[s].y, gv[s].y),
                               __fadd_rn(ev[s].z, gv[s].z), __fadd_rn(ev[s].w, gv[s].w));
        } else {
            p[s] = gv[s];
        }
    }
}

template <int SCHEME>
__device__ __forceinline__ void accumulate_slots(Stats<SCHEME> &st, uint32_t w0, int tt,
                                                 int team_threads, uint32_t cnt,
                                                 const float4 (&p)[kSlots]) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = w0 + static_cast<uint32_t>(s * team_threads + tt) * 4u;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (j + c < cnt) st.add(get(p[s], c));
    }
}

template <int SCHEME, int BITS, bool SR, bool EF>
__device__ __forceinline__ void quantize_slots(const EncodeParams &P, uint64_t b0, uint32_t cnt,
                                               uint32_t w0, int tt, int team_threads, int lane,
                                               const float4 (&p)[kSlots],
                                               const bool (&full)[kSlots],
                                               const BucketParams &bp) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = w0 + static_cast<uint32_t>(s * team_threads + tt) * 4u;
        const uint64_t i = b0 + j;
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (SR) {
            if (j < cnt) uniform4(i, P.seed, P.step, u);
        }
        uint32_t field = 0;
        float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (j + c < cnt) {
                float deq;
                const float pc = get(p[s], c);
                const uint32_t q = quantize<SCHEME, BITS, SR>(pc, u[c], bp, deq);
                field |= q << (c * BITS);
                set(e, c, __fsub_rn(pc, deq));
            }
        }
        const uint32_t word = gather_word<BITS>(field);
        if (j < cnt && stores_word<BITS>(lane)) __stcs(P.codes + (i * BITS) / 32u, word);
        if constexpr (EF) {
            if (full[s]) {
                __stcs(reinterpret_cast<float4 *>(P.err + i), e);
            } else if (j < cnt) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (j + c < cnt) P.err[i + c] = get(e, c);
            }
        }
    }
}

template <int SCHEME, int BITS, bool SR, typename TIn, bool EF>
__global__ void __launch_bounds__(kBlock) encode_kernel(const EncodeParams P) {
    __shared__ Stats<SCHEME> red[2][kBlock / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint32_t window = static_cast<uint32_t>(kWindowPerWarp * W);
    const uint64_t ngroups = (P.nbuckets + teams - 1) / teams;
    int buf = 0;

    for (uint64_t grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
        const uint64_t k = grp * teams + team;
        const bool active = k < P.nbuckets;
        const uint64_t b0 = k * P.bucket;
        const uint32_t cnt =
            active ? static_cast<uint32_t>(min(static_cast<uint64_t>(P.bucket), P.n - b0)) : 0u;

        float4 p[kSlots];
        bool full[kSlots];
        Stats<SCHEME> st;
        st.init();
        if (!P.two_pass) {
            load_slots<TIn, EF>(P, b0, cnt, 0u, tt, team_threads, p, full);
            accumulate_slots<SCHEME>(st, 0u, tt, team_threads, cnt, p);
        } else {
            for (uint32_t w0 = 0; w0 < cnt; w0 += window) {
                load_slots<TIn, EF>(P, b0, cnt, w0, tt, team_threads, p, full);
                accumulate_slots<SCHEME>(st, w0, tt, team_threads, cnt, p);
            }
        }
        st.warp_reduce();
        if (W > 1) {
            if (lane == 0) red[buf][warp] = st;
            __syncthreads();
            st = red[buf][team * W];
            for (int w = 1; w < W; ++w) st.merge(red[buf][team * W + w]);
            buf ^= 1;
        }
        const BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);

        if (!P.two_pass) {
            quantize_slots<SCHEME, BITS, SR, EF>(P, b0, cnt, 0u, tt, team_threads, lane, p, full,
                                                 bp);
        } else {
            for (uint32_t w0 = 0; w0 < cnt; w0 += window) {
                load_slots<TIn, EF>(P, b0, cnt, w0, tt, team_threads, p, full);
                quantize_slots<SCHEME, BITS, SR, EF>(P, b0, cnt, w0, tt, team_threads, lane, p,
                                                     full, bp);
            }
        }
        if (active && tt == 0) {
            if constexpr (SCHEME == kUniform) {
                P.scale[k] = bp.scale;
                P.offset[k] = bp.a;
            } else {
                P.scale[k] = bp.a;
            }
        }
    }
}

template <int SCHEME, int BITS, bool SR, typename TIn, bool EF>
cudaError_t launch_one(const EncodeParams &p, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&encode_kernel<SCHEME, BITS, SR, TIn, EF>);
    const int teams = (kBlock / 32) / p.team_warps;
    const uint64_t groups = (p.nbuckets + teams - 1) / teams;
    const int grid = persistent_grid(fn, kBlock, groups);
    encode_kernel<SCHEME, BITS, SR, TIn, EF><<<grid, kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int SCHEME, int BITS, bool SR>
cudaError_t launch_dtype(const EncodeParams &p, int bf16, cudaStream_t stream) {
    const bool ef = p.err != nullptr;
    if (bf16)
        return ef ? launch_one<SCHEME, BITS, SR, uint16_t, true>(p, stream)
                  : launch_one<SCHEME, BITS, SR, uint16_t, false>(p, stream);
    return ef ? launch_one<SCHEME, BITS, SR, float, true>(p, stream)
              : launch_one<SCHEME, BITS, SR, float, false>(p, stream);
}

template <int SCHEME, int BITS>
cudaError_t launch_round(const EncodeParams &p, int stochastic, int bf16, cudaStream_t stream) {
    return stochastic ? launch_dtype<SCHEME, BITS, true>(p, bf16, stream)
                      : launch_dtype<SCHEME, BITS, false>(p, bf16, stream);
}

}  // namespace

cudaError_t launch_encode(const EncodeParams &p, int scheme, int bits, int stochastic, int bf16,
                          cudaStream_t stream) {
    if (scheme == kSign) return launch_dtype<kSign, 1, false>(p, bf16, stream);
    if (scheme == kTernary) return launch_round<kTernary, 2>(p, stochastic, bf16, stream);
    switch (bits) {
        case 1: return launch_round<kUniform, 1>(p, stochastic, bf16, stream);
        case 2: return launch_round<kUniform, 2>(p, stochastic, bf16, stream);
        case 4: return launch_round<kUniform, 4>(p, stochastic, bf16, stream);
        default: return launch_round<kUniform, 8>(p, stochastic, bf16, stream);
    }
}

}  // namespace qc
