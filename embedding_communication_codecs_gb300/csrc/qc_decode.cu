// qc_decode.cu -- receiver half of the codec: dequantize M workers' payloads and
// accumulate them in fp32 in a fixed worker order; signSGD majority vote.
//
// "Quantization for Communication", "Quantization-Aware All-Reduce" (dequantize
// after the exchange, accumulate in higher precision) and "Quantized SGD
// Algorithms" (SignSGD aggregates by majority vote); "Gradient Compression and
// Quantised Collectives", "Why sparsification fights the all-reduce".
//
// Decode layout: one warp owns one bucket at a time, so the bucket index and the
// per-worker scale/offset are known without any per-element division.  Lane l
// of slot s covers elements (s * 32 + l) * 4 .. +3 of a 512-element window: the
// fp32 output is written as lane-contiguous float4s (fully coalesced), and each
// worker's codes for those four elements are one 4*b-bit field.
#include "qc_decode_math.cuh"

namespace qc {
namespace {

// The 4*BITS-bit field holding the codes of elements i .. i+3 (i % 4 == 0).
template <int BITS>
__device__ __forceinline__ uint32_t load_field(const uint32_t *words, uint64_t i) {
    if constexpr (BITS == 8) {
        return __ldcs(words + (i >> 2));
    } else if constexpr (BITS == 4) {
        return __ldcs(reinterpret_cast<const unsigned short *>(words) + (i >> 2));
    } else if constexpr (BITS == 2) {
        return __ldcs(reinterpret_cast<const unsigned char *>(words) + (i >> 2));
    } else {
        const uint32_t byte = __ldcs(reinterpret_cast<const unsigned char *>(words) + (i >> 3));
        return (byte >> (((i >> 2) & 1u) * 4u)) & 0xFu;
    }
}

// The outputs of one window (4 per lane and slot) from the accumulated values:
// MEAN and accumulate flags, then the stores.
__device__ __forceinline__ void store_window(const DecodeParams &P, float (&acc)[kSlots][4],
                                             uint64_t b0, uint32_t w0, uint32_t cnt, int lane,
                                             float Mf) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = w0 + static_cast<uint32_t>(s * 32 + lane) * 4u;
        if (j >= cnt) continue;
        const uint64_t i = b0 + j;
        float4 r = make_float4(acc[s][0], acc[s][1], acc[s][2], acc[s][3]);
        if (P.flags & 1) {
            r = P.inv_m != 0.0f
                    ? make_float4(__fmul_rn(r.x, P.inv_m), __fmul_rn(r.y, P.inv_m),
                                  __fmul_rn(r.z, P.inv_m), __fmul_rn(r.w, P.inv_m))
                    : make_float4(__fdiv_rn(r.x, Mf), __fdiv_rn(r.y, Mf),
                                  __fdiv_rn(r.z, Mf), __fdiv_rn(r.w, Mf));
        }
        if (j + 4u <= cnt) {
            float4 *o = reinterpret_cast<float4 *>(P.out + i);
            if (P.flags & 2) {
                const float4 prev = __ldcs(o);
                r = make_float4(__fadd_rn(prev.x, r.x), __fadd_rn(prev.y, r.y),
                                __fadd_rn(prev.z, r.z), __fadd_rn(prev.w, r.w));
            }
            __stcs(o, r);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j + c < cnt) {
                    float v = get(r, c);
                    if (P.flags & 2) v = __fadd_rn(P.out[i + c], v);
                    P.out[i + c] = v;
                }
            }
        }
    }
}

// One worker (M = 1): a warp's items are (bucket, window) pairs, and the code
// fields, scale and offset of its next item are loaded before the current one
// is dequantized and stored, so that a load is in flight while the warp works.
template <int SCHEME, int BITS>
__device__ __forceinline__ void decode_single(const DecodeParams &P, int lane, uint64_t first,
                                              uint64_t warps) {
    const uint32_t wpb = (static_cast<uint32_t>(P.bucket) + kWindowPerWarp - 1u) / kWindowPerWarp;
    const uint64_t items = P.nbuckets * wpb;
    const float Mf = 1.0f;
    uint32_t f[kSlots];
    float sc = 0.0f, of = 0.0f;
    uint64_t b0 = 0;
    uint32_t w0 = 0, cnt = 0;
    auto load = [&](uint64_t t, uint32_t (&fd)[kSlots], float &s_, float &o_, uint64_t &b0_,
                    uint32_t &w0_, uint32_t &cnt_) {
        const uint64_t k = t / wpb;
        w0_ = static_cast<uint32_t>(t - k * wpb) * kWindowPerWarp;
        b0_ = k * P.bucket;
        cnt_ = static_cast<uint32_t>(min(static_cast<uint64_t>(P.bucket), P.n - b0_));
        s_ = __ldg(P.scale + k);
        o_ = 0.0f;
        if constexpr (SCHEME == kUniform) o_ = __ldg(P.offset + k);
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const uint32_t j = w0_ + static_cast<uint32_t>(s * 32 + lane) * 4u;
            fd[s] = (j < cnt_) ? load_field<BITS>(P.codes, b0_ + j) : 0u;
        }
    };
    if (first < items) load(first, f, sc, of, b0, w0, cnt);
    for (uint64_t t = first; t < items; t += warps) {
        uint32_t fn[kSlots];
        float scn = 0.0f, ofn = 0.0f;
        uint64_t b0n = 0;
        uint32_t w0n = 0, cntn = 0;
        if (t + warps < items) load(t + warps, fn, scn, ofn, b0n, w0n, cntn);
        float acc[kSlots][4];
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[s][c] = accumulate_code<SCHEME, BITS>(0.0f, f[s], c, sc, of);
        store_window(P, acc, b0, w0, cnt, lane, Mf);
#pragma unroll
        for (int s = 0; s < kSlots; ++s) f[s] = fn[s];
        sc = scn;
        of = ofn;
        b0 = b0n;
        w0 = w0n;
        cnt = cntn;
    }
}

template <int SCHEME, int BITS>
__global__ void __launch_bounds__(kBlock) decode_kernel(const __grid_constant__ DecodeParams P) {
    const int lane = threadIdx.x & 31;
    const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (kBlock / 32);
    const float Mf = static_cast<float>(P.M);
    // (QSGD keeps the plain loop: measured slower with the prefetch)
    if (SCHEME != kQsgd && P.M == 1) {
        decode_single<SCHEME, BITS>(P, lane, static_cast<uint64_t>(blockIdx.x) * (kBlock / 32) + (threadIdx.x >> 5),
                                    warps);
        return;
    }

    for (uint64_t k = static_cast<uint64_t>(blockIdx.x) * (kBlock / 32) + (threadIdx.x >> 5);
         k < P.nbuckets; k += warps) {
        const uint64_t b0 = k * P.bucket;
        const uint32_t cnt = static_cast<uint32_t>(min(static_cast<uint64_t>(P.bucket), P.n - b0));
        for (uint32_t w0 = 0; w0 < cnt; w0 += kWindowPerWarp) {
            float acc[kSlots][4];
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[s][c] = 0.0f;

#pragma unroll 2
            for (int w = 0; w < P.M; ++w) {
                const uint32_t *cw = P.codes + static_cast<uint64_t>(w) * P.codes_stride;
                const float sc = __ldg(P.scale + static_cast<uint64_t>(w) * P.meta_stride + k);
                float of = 0.0f;
                if constexpr (SCHEME == kUniform)
                    of = __ldg(P.offset + static_cast<uint64_t>(w) * P.meta_stride + k);
                uint32_t field[kSlots];
#pragma unroll
                for (int s = 0; s < kSlots; ++s) {
                    const uint32_t j = w0 + static_cast<uint32_t>(s * 32 + lane) * 4u;
                    field[s] = (j < cnt) ? load_field<BITS>(cw, b0 + j) : 0u;
                }
#pragma unroll
                for (int s = 0; s < kSlots; ++s)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[s][c] = accumulate_code<SCHEME, BITS>(acc[s][c], field[s], c, sc, of);
            }

            store_window(P, acc, b0, w0, cnt, lane, Mf);
        }
    }
}

template <int SCHEME, int BITS>
cudaError_t launch_decode_one(const DecodeParams &p, cudaStream_t stream) {
    const void *fn = reinterpret_cast<const void *>(&decode_kernel<SCHEME, BITS>);
    const uint64_t blocks = (p.nbuckets + (kBlock / 32) - 1) / (kBlock / 32);
    const int grid = persistent_grid(fn, kBlock, blocks);
    decode_kernel<SCHEME, BITS><<<grid, kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

// ----------------------------------------------------------------- sign vote
//
// Bit-sliced vertical counter: plane j holds bit j of every column's count.
// Adding one worker's word ripples a carry through the planes (two logic ops
// per plane); NP planes count up to 2^NP - 1 workers.  The comparison
// count >= threshold is evaluated plane by plane from the top.

template <int NP>
__device__ __forceinline__ void count_add(uint32_t (&pl)[NP], uint32_t x) {
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const uint32_t carry = pl[j] & x;
        pl[j] ^= x;
        x = carry;
    }
}

template <int NP>
__device__ __forceinline__ uint32_t count_ge(const uint32_t (&pl)[NP], uint32_t threshold) {
    uint32_t gt = 0u, eq = 0xFFFFFFFFu;
#pragma unroll
    for (int j = NP - 1; j >= 0; --j) {
        if ((threshold >> j) & 1u) {
            eq &= pl[j];
        } else {
            gt |= eq & pl[j];
            eq &= ~pl[j];
        }
    }
    return gt | eq;
}

template <int NP, bool VEC>
__global__ void __launch_bounds__(kBlock) vote_kernel(const VoteParams P) {
    constexpr int kWords = VEC ? 4 : 1;
    const uint64_t groups = (P.nwords + kWords - 1) / kWords;
    for (uint64_t g = static_cast<uint64_t>(blockIdx.x) * kBlock + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * kBlock) {
        const uint64_t w0 = g * kWords;
        uint32_t pl[kWords][NP];
#pragma unroll
        for (int c = 0; c < kWords; ++c)
#pragma unroll
            for (int j = 0; j < NP; ++j) pl[c][j] = 0u;
        const bool whole = w0 + kWords <= P.nwords;
#pragma unroll 4
        for (int w = 0; w < P.M; ++w) {
            const uint32_t *src = P.signs + static_cast<uint64_t>(w) * P.stride + w0;
            uint32_t x[kWords];
            if constexpr (VEC) {
                if (whole) {
                    const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(src));
                    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
                } else {
#pragma unroll
                    for (int c = 0; c < kWords; ++c)
                        x[c] = (w0 + c < P.nwords) ? __ldcs(src + c) : 0u;
                }
            } else {
                x[0] = __ldcs(src);
            }
#pragma unroll
            for (int c = 0; c < kWords; ++c) count_add<NP>(pl[c], x[c]);
        }
        uint32_t r[kWords];
#pragma unroll
        for (int c = 0; c < kWords; ++c) {
            r[c] = count_ge<NP>(pl[c], P.threshold);
            if (w0 + c == P.nwords - 1) r[c] &= P.last_mask;
        }
        if constexpr (VEC) {
            if (whole) {
                __stcs(reinterpret_cast<uint4 *>(P.out + w0), make_uint4(r[0], r[1], r[2], r[3]));
            } else {
#pragma unroll
                for (int c = 0; c < kWords; ++c)
                    if (w0 + c < P.nwords) P.out[w0 + c] = r[c];
            }
        } else {
            P.out[w0] = r[0];
        }
    }
}

template <int NP>
cudaError_t launch_vote_np(const VoteParams &p, bool vec, cudaStream_t stream) {
    const int words = vec ? 4 : 1;
    const uint64_t groups = (p.nwords + words - 1) / words;
    const uint64_t blocks = (groups + kBlock - 1) / kBlock;
    if (vec) {
        const int grid = persistent_grid(reinterpret_cast<const void *>(&vote_kernel<NP, true>),
                                         kBlock, blocks);
        vote_kernel<NP, true><<<grid, kBlock, 0, stream>>>(p);
    } else {
        const int grid = persistent_grid(reinterpret_cast<const void *>(&vote_kernel<NP, false>),
                                         kBlock, blocks);
        vote_kernel<NP, false><<<grid, kBlock, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int scheme, int bits, cudaStream_t stream) {
    if (scheme == kSign) return launch_decode_one<kSign, 1>(p, stream);
    if (scheme == kTernary) return launch_decode_one<kTernary, 2>(p, stream);
    if (scheme == kLog) {
        if (bits == 2) return launch_decode_one<kLog, 2>(p, stream);
        if (bits == 4) return launch_decode_one<kLog, 4>(p, stream);
        return launch_decode_one<kLog, 8>(p, stream);
    }
    if (scheme == kQsgd) {
        if (bits == 2) return launch_decode_one<kQsgd, 2>(p, stream);
        if (bits == 4) return launch_decode_one<kQsgd, 4>(p, stream);
        return launch_decode_one<kQsgd, 8>(p, stream);
    }
    switch (bits) {
        case 1: return launch_decode_one<kUniform, 1>(p, stream);
        case 2: return launch_decode_one<kUniform, 2>(p, stream);
        case 4: return launch_decode_one<kUniform, 4>(p, stream);
        default: return launch_decode_one<kUniform, 8>(p, stream);
    }
}

cudaError_t launch_vote(const VoteParams &p, bool vec, cudaStream_t stream) {
    int np = 0;
    while ((1 << np) <= p.M) ++np;  // planes to count 0 .. M
    switch (np) {
        case 1: return launch_vote_np<1>(p, vec, stream);
        case 2: return launch_vote_np<2>(p, vec, stream);
        case 3: return launch_vote_np<3>(p, vec, stream);
        case 4: return launch_vote_np<4>(p, vec, stream);
        case 5: return launch_vote_np<5>(p, vec, stream);
        case 6: return launch_vote_np<6>(p, vec, stream);
        case 7: return launch_vote_np<7>(p, vec, stream);
        case 8: return launch_vote_np<8>(p, vec, stream);
        case 9: return launch_vote_np<9>(p, vec, stream);
        case 10: return launch_vote_np<10>(p, vec, stream);
        default: return launch_vote_np<11>(p, vec, stream);
    }
}

}  // namespace qc
