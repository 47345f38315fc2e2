// qc_encode_direct.cuh -- the direct (register-staged) encode kernel template:
// error-feedback quantization of a flat gradient, one single-pass kernel per
// (scheme, bits, rounding, dtype, EF).  Included by the translation units that
// instantiate it (qc_encode.cu, qc_encode_direct_log.cu).
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
#pragma once

#include "qc_encode_math.cuh"

namespace qc {
namespace {

// --------------------------------------------------------------- the kernel

// p = e + g for the lane's slots of the window of `wcnt` valid elements
// starting at global element `base`.
template <typename TIn, bool EF>
__device__ __forceinline__ void load_slots(const EncodeParams &P, uint64_t base, uint32_t wcnt,
                                           int tt, int team_threads, float4 (&p)[kSlots]) {
    const TIn *g = static_cast<const TIn *>(P.grad);
    float4 gv[kSlots], ev[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u;
        const uint64_t i = base + j;
        gv[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        ev[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j + 4u <= wcnt) {
            gv[s] = GradLoad<TIn>::full(g, i);
            if constexpr (EF) ev[s] = __ldcs(reinterpret_cast<const float4 *>(P.err + i));
        } else if (j < wcnt) {  // ragged end of the array: element-wise
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j + c < wcnt) {
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

template <int SCHEME, int BITS, bool SR, typename TIn, bool EF>
__global__ void __launch_bounds__(kBlock) encode_kernel(const __grid_constant__ EncodeParams P) {
    __shared__ Stats<SCHEME> red[2][kBlock / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint32_t window = static_cast<uint32_t>(kWindowPerWarp * W);
    const uint64_t ngroups = (P.nbuckets + teams - 1) / teams;
    const PhiloxKeys &keys = P.keys;
    int buf = 0;

    for (uint64_t grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
        const uint64_t k = grp * teams + team;
        const bool active = k < P.nbuckets;
        const uint64_t b0 = k * P.bucket;
        const uint32_t cnt =
            active ? static_cast<uint32_t>(min(static_cast<uint64_t>(P.bucket), P.n - b0)) : 0u;

        float4 p[kSlots];
        Stats<SCHEME> st;
        st.init();
        if (!P.two_pass) {
            load_slots<TIn, EF>(P, b0, cnt, tt, team_threads, p);
            accumulate_slots<SCHEME>(st, p, tt, team_threads, cnt);
        } else {
            for (uint32_t w0 = 0; w0 < cnt; w0 += window) {
                load_slots<TIn, EF>(P, b0 + w0, cnt - w0, tt, team_threads, p);
                accumulate_slots<SCHEME>(st, p, tt, team_threads, cnt - w0);
            }
        }
        team_reduce<SCHEME>(st, red, buf, W, warp, lane, team);
        BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);
        if constexpr (SCHEME == kQsgd) {
            if (bp.exact) {  // rare: the norm next to a rounding boundary (uniform per team)
                WideSum acc;
                wide_zero(acc);
                if (!P.two_pass) {
                    wide_add_slots(acc, p, tt, team_threads, cnt);
                } else {
                    for (uint32_t w0 = 0; w0 < cnt; w0 += window) {
                        load_slots<TIn, EF>(P, b0 + w0, cnt - w0, tt, team_threads, p);
                        wide_add_slots(acc, p, tt, team_threads, cnt - w0);
                    }
                }
                bp = qsgd_params<BITS>(team_exact_norm<SCHEME, 1>(acc, red, W, warp, lane, team));
            }
        }

        if (!P.two_pass) {
            quantize_store_slots<SCHEME, BITS, SR, EF>(P.codes, P.err, b0, cnt, tt, team_threads,
                                                       lane, p, bp, P.step, keys, P.index_base);
        } else {
            for (uint32_t w0 = 0; w0 < cnt; w0 += window) {
                load_slots<TIn, EF>(P, b0 + w0, cnt - w0, tt, team_threads, p);
                quantize_store_slots<SCHEME, BITS, SR, EF>(P.codes, P.err, b0 + w0, cnt - w0, tt,
                                                           team_threads, lane, p, bp, P.step,
                                                           keys, P.index_base);
            }
        }
        if (active && tt == 0) store_meta<SCHEME>(P.scale, P.offset, k, bp);
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
}  // namespace qc
