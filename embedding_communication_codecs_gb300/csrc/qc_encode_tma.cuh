// qc_encode_tma.cuh -- the encode kernel template with the gradient (and
// residual) streamed through a multi-stage shared-memory pipeline by TMA bulk
// copies.  Included by the translation units that instantiate it
// (qc_encode_tma.cu, qc_encode_clip.cu); each keeps its own error flag.
//
// "Quantization for Communication", "Quantization Schemes", "Quantized SGD
// Algorithms", "Error Feedback for Quantization", "Hardware Acceleration" (the
// arithmetic is the shared code in qc_encode_math.cuh).
//
// A tile is TB whole buckets (TE = TB * bucket elements, about 24-32 KB of
// input).  Each persistent block owns tiles blockIdx.x, blockIdx.x + grid, ...;
// thread 0 keeps `stages - 1` tiles of copies in flight ahead of the one being
// quantized, so the bytes in flight per SM no longer depend on registers.  The
// compute side is the team layout of the direct kernel, reading its slots from
// shared memory; codes, residuals and metadata are stored straight from
// registers.  Tail bytes that are not a whole 16-byte unit (n % 4 != 0 for
// fp32) are read from global memory directly.
#pragma once

#include "qc_encode_math.cuh"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_encode_errors;

namespace {

// The segment that owns launch tile `tile` (binary search on the segments'
// first tiles, which ascend).
__device__ __forceinline__ uint32_t segment_of(const EncodeSegs &S, uint64_t tile) {
    uint32_t lo = 0, hi = S.nseg;
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        if (S.s[mid].tile0 <= tile) lo = mid;
        else hi = mid;
    }
    return lo;
}

// The bulk copies of tile `lt` of one segment (lt counted within the segment).
template <typename TIn, bool EF>
__device__ __forceinline__ void issue_seg_tile(const EncodeSeg &sg, const EncodeTiles &G,
                                               uint64_t lt, unsigned char *stage, uint64_t *bar) {
    const uint64_t t0 = lt * G.te;
    const uint64_t tcnt = min(static_cast<uint64_t>(G.te), sg.n - t0);
    const uint32_t gb = floor16(tcnt * sizeof(TIn));
    const uint32_t eb = EF ? floor16(tcnt * 4u) : 0u;
    mbar_arrive_expect_tx(bar, gb + eb);
    if (gb) bulk_load(stage, static_cast<const TIn *>(sg.grad) + t0, gb, bar);
    if (EF && eb) bulk_load(stage + G.e_offset, sg.err + t0, eb, bar);
}

template <typename TIn, bool EF>
__device__ __forceinline__ void issue_tile(const EncodeSegs &S, const EncodeTiles &G,
                                           uint64_t tile, unsigned char *stage, uint64_t *bar) {
    const EncodeSeg &sg = S.s[segment_of(S, tile)];
    issue_seg_tile<TIn, EF>(sg, G, tile - sg.tile0, stage, bar);
}

// Elements of the tile that the bulk copies brought into shared memory.
template <typename TIn, bool EF>
__device__ __forceinline__ uint32_t staged_elems(uint32_t tcnt) {
    uint32_t g = floor16(static_cast<uint64_t>(tcnt) * sizeof(TIn)) / sizeof(TIn);
    if constexpr (EF) g = min(g, floor16(static_cast<uint64_t>(tcnt) * 4u) / 4u);
    return g;
}

template <typename TIn>
__device__ __forceinline__ float4 smem_grad4(const unsigned char *stage, uint32_t e) {
    if constexpr (sizeof(TIn) == 4) {
        return *reinterpret_cast<const float4 *>(stage + e * 4u);
    } else {
        return unpack_bf16x4(*reinterpret_cast<const uint2 *>(stage + e * 2u));
    }
}

template <typename TIn>
__device__ __forceinline__ float smem_grad1(const unsigned char *stage, uint32_t e) {
    if constexpr (sizeof(TIn) == 4) {
        return *reinterpret_cast<const float *>(stage + e * 4u);
    } else {
        return bf16_bits_to_float(*reinterpret_cast<const unsigned short *>(stage + e * 2u));
    }
}

// p = e + g for the lane's slots of the bucket at tile offset b_off.  FULL: every
// slot is valid and staged.
template <typename TIn, bool EF, bool FULL = false>
__device__ __forceinline__ void load_slots_staged(const EncodeSeg &P, const EncodeTiles &G,
                                                  const unsigned char *stage, uint64_t t0,
                                                  uint32_t b_off, uint32_t cnt, uint32_t staged,
                                                  int tt, int team_threads,
                                                  float4 (&p)[kSlots]) {
    const TIn *g = static_cast<const TIn *>(P.grad);
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u;
        const uint32_t e = b_off + j;
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f), ev = gv;
        if (FULL || (j + 4u <= cnt && e + 4u <= staged)) {
            gv = smem_grad4<TIn>(stage, e);
            if constexpr (EF) ev = *reinterpret_cast<const float4 *>(stage + G.e_offset + e * 4u);
        } else if (j < cnt) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (j + c < cnt) {
                    if (e + c < staged) {
                        set(gv, c, smem_grad1<TIn>(stage, e + c));
                        if constexpr (EF)
                            set(ev, c, *reinterpret_cast<const float *>(stage + G.e_offset +
                                                                        (e + c) * 4u));
                    } else {
                        set(gv, c, GradLoad<TIn>::one(g, t0 + e + c));
                        if constexpr (EF) set(ev, c, P.err[t0 + e + c]);
                    }
                }
            }
        }
        if constexpr (EF) {
            p[s] = make_float4(__fadd_rn(ev.x, gv.x), __fadd_rn(ev.y, gv.y), __fadd_rn(ev.z, gv.z),
                               __fadd_rn(ev.w, gv.w));
        } else {
            p[s] = gv;
        }
    }
}

template <int SCHEME, int BITS, bool SR, typename TIn, bool EF>
__global__ void __launch_bounds__(kBlock) encode_tma_kernel(const __grid_constant__ EncodeParams P,
                                                            const __grid_constant__ EncodeTiles G,
                                                            const __grid_constant__ EncodeSegs S) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G.stages * G.stage_bytes);
    auto red = reinterpret_cast<Stats<SCHEME>(*)[kBlock / 32]>(full + G.stages);
    uint32_t *hist = reinterpret_cast<uint32_t *>(red + 2);  // CLIP: the teams' histograms

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint32_t window = static_cast<uint32_t>(team_threads) * kSlots * 4u;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    if constexpr (SCHEME == kClip) {
        for (int i = threadIdx.x; i < teams * sel_region_words(P.bucket); i += kBlock) hist[i] = 0u;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) {
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(s) * gridDim.x;
            if (tile < G.ntiles)
                issue_tile<TIn, EF>(S, G, tile, smem + s * G.stage_bytes, &full[s]);
        }
    }

    int buf = 0;
    uint32_t sel_parity = 0;  // CLIP: which histogram set the team's next bucket uses
    uint32_t it = 0;
    bool failed = false;
    for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % G.stages;
        const unsigned char *stage = smem + s * G.stage_bytes;
        // Each thread waits for the stage on its own.  A team learns whether
        // all of its waits succeeded from the reduction of its statistics (the
        // warp's vote, or the block barrier that a multi-warp team's exchange
        // takes anyway), before it stores anything: a team that learns of a
        // timeout stores no codes, metadata or residual for the tile.  The
        // block learns it at the one barrier per tile below, which also frees
        // the stage for its refill, and stops there.  (A separate agreement
        // barrier before the compute measured 7 % slower on the 4-bit encode.)
        const bool ok = mbar_wait(&full[s], (it / G.stages) & 1u);

        const EncodeSeg &sg = S.s[segment_of(S, tile)];
        const uint64_t lt = tile - sg.tile0;  // the tile within its segment
        const PhiloxKeys &keys = P.keys;
        const uint64_t t0 = lt * G.te;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(G.te), sg.n - t0));
        const uint32_t staged = staged_elems<TIn, EF>(tcnt);
        for (uint32_t kb0 = 0; kb0 < G.tb; kb0 += teams) {
            const uint32_t kb = kb0 + team;
            const uint32_t b_off = kb * P.bucket;
            const uint32_t cnt = (kb < G.tb && b_off < tcnt) ? min(P.bucket, tcnt - b_off) : 0u;
            // a bucket that fills the team's window and is wholly staged takes
            // the path without per-slot bounds checks (uniform across the team)
            const bool whole = cnt == window && b_off + cnt <= staged;
            float4 p[kSlots];
            Stats<SCHEME> st;
            st.init();
            if (whole) {
                load_slots_staged<TIn, EF, true>(sg, G, stage, t0, b_off, cnt, staged, tt,
                                                 team_threads, p);
                if constexpr (SCHEME != kClip) accumulate_slots<SCHEME, true>(st, p, tt, team_threads, cnt);
            } else {
                load_slots_staged<TIn, EF>(sg, G, stage, t0, b_off, cnt, staged, tt, team_threads, p);
                if constexpr (SCHEME != kClip) accumulate_slots<SCHEME>(st, p, tt, team_threads, cnt);
            }
            bool team_ok;
            if constexpr (SCHEME == kClip) {
                team_ok = __syncthreads_and(ok) != 0;  // the selection has no block barrier of its own
                uint32_t *region = hist + team * sel_region_words(P.bucket);
                if (whole)
                    team_percentiles<true>(p, cnt, P.bucket, tt, team_threads, W, team, warp % W,
                                           lane, region, sel_parity, st.mn, st.mx);
                else if (cnt)
                    team_percentiles<false>(p, cnt, P.bucket, tt, team_threads, W, team, warp % W,
                                            lane, region, sel_parity, st.mn, st.mx);
            } else {
                team_ok = team_reduce_ok<SCHEME>(st, red, buf, W, warp, lane, team, ok);
            }
            BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);
            if constexpr (SCHEME == kQsgd) {
                if (bp.exact) {  // rare: the norm next to a rounding boundary (uniform per team)
                    bp = qsgd_params<BITS>(team_exact_norm_slots<SCHEME, 1>(p, tt, team_threads, cnt,
                                                                            red, W, warp, lane, team));
                }
            }
            if (!team_ok) continue;  // a wait timed out: store nothing (the block stops below)
            if (whole)
                quantize_store_slots<SCHEME, BITS, SR, EF, true>(sg.codes, sg.err, t0 + b_off, cnt, tt,
                                                                 team_threads, lane, p, bp, P.step,
                                                                 keys, sg.index_base);
            else
                quantize_store_slots<SCHEME, BITS, SR, EF>(sg.codes, sg.err, t0 + b_off, cnt, tt,
                                                           team_threads, lane, p, bp, P.step, keys,
                                                           sg.index_base);
            if (cnt && tt == 0) store_meta<SCHEME>(sg.scale, sg.offset, lt * G.tb + kb, bp);
        }
        // Every thread is done with this stage, and every wait succeeded, before
        // the stage is refilled.
        if (!__syncthreads_and(ok)) {
            failed = true;
            break;
        }
        if (threadIdx.x == 0) {
            const uint64_t next = tile + static_cast<uint64_t>(G.stages) * gridDim.x;
            if (next < G.ntiles)
                issue_tile<TIn, EF>(S, G, next, smem + s * G.stage_bytes, &full[s]);
        }
    }
    if (failed && threadIdx.x == 0) {
        report_failure(&g_encode_errors, P.status, kErrPipelineTimeout);
        // Let every copy this block may still have in flight land (bounded).
        for (uint32_t d = 0; d < G.stages; ++d) {
            const uint32_t j = it + d;
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
            if (tile < G.ntiles) mbar_wait(&full[j % G.stages], (j / G.stages) & 1u);
        }
    }
}

template <int SCHEME, int BITS, bool SR, typename TIn, bool EF>
cudaError_t launch_one(const EncodeParams &p, const EncodeTiles &g, cudaStream_t stream,
                       const EncodeSegs *segs) {
    auto fn = &encode_tma_kernel<SCHEME, BITS, SR, TIn, EF>;
    size_t smem = encode_tiles_smem(g, sizeof(Stats<SCHEME>));
    if (SCHEME == kClip)
        smem += static_cast<size_t>((kBlock / 32) / p.team_warps) * sel_region_words(p.bucket) * 4u;
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kBlock, g.ntiles, smem);
    if (segs) fn<<<grid, kBlock, smem, stream>>>(p, g, *segs);
    else fn<<<grid, kBlock, smem, stream>>>(p, g, single_segment(p));
    return cudaGetLastError();
}

template <int SCHEME, int BITS, bool SR>
cudaError_t launch_dtype(const EncodeParams &p, const EncodeTiles &g, int bf16,
                         cudaStream_t stream, const EncodeSegs *segs) {
    const bool ef = p.err != nullptr;
    if (bf16)
        return ef ? launch_one<SCHEME, BITS, SR, uint16_t, true>(p, g, stream, segs)
                  : launch_one<SCHEME, BITS, SR, uint16_t, false>(p, g, stream, segs);
    return ef ? launch_one<SCHEME, BITS, SR, float, true>(p, g, stream, segs)
              : launch_one<SCHEME, BITS, SR, float, false>(p, g, stream, segs);
}

template <int SCHEME, int BITS>
cudaError_t launch_round(const EncodeParams &p, const EncodeTiles &g, int stochastic, int bf16,
                         cudaStream_t stream, const EncodeSegs *segs = nullptr) {
    return stochastic ? launch_dtype<SCHEME, BITS, true>(p, g, bf16, stream, segs)
                      : launch_dtype<SCHEME, BITS, false>(p, g, bf16, stream, segs);
}

}  // namespace
}  // namespace qc
