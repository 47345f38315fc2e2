// qc_reencode.cuh -- the fused receiver re-encode kernel template, included by
// the translation units that instantiate it (qc_reencode.cu: the uniform
// scheme; qc_reencode_other.cu: sign, ternary and QSGD); each keeps its own
// error flag.  The method and the kernel design are described in qc_reencode.cu.
#pragma once

#include "qc_encode_math.cuh"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_reencode_errors;

namespace {

constexpr int kReBlock = kProducerBlock;
constexpr int kConsumers = kConsumerWarps * 32;
static_assert(kConsumers == kBlock, "the encode teams span exactly the consumer warps");

__device__ __forceinline__ float finish_r(float a, const ReencodeParams &P, float Mf) {
    if (P.flags & 1) return P.inv_m != 0.0f ? __fmul_rn(a, P.inv_m) : __fdiv_rn(a, Mf);
    return a;
}

// The lane's slots of the bucket window [w0, w0 + cnt) at tile offset b_off,
// read from the sum buffer (zeros past cnt).  FULL: every slot is valid.
template <bool FULL = false>
__device__ __forceinline__ void load_slots_sum(const float *pb, uint32_t b_off, uint32_t cnt,
                                               int tt, int team_threads, float4 (&p)[kSlots]) {
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const uint32_t j = static_cast<uint32_t>(s * team_threads + tt) * 4u;
        if (FULL || j + 4u <= cnt) {
            p[s] = *reinterpret_cast<const float4 *>(pb + b_off + j);
        } else {
            p[s] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (j + c < cnt) set(p[s], c, pb[b_off + j + c]);
        }
    }
}

template <int SCHEME, int BITS, bool SR, bool EF>
__global__ void __launch_bounds__(kReBlock, 2) reencode_kernel(const __grid_constant__ ReencodeParams P,
                                                               const __grid_constant__ ReencodeTiles G) {
    extern __shared__ __align__(128) unsigned char smem[];
    float *sums = reinterpret_cast<float *>(smem + G.stages * G.stage_bytes);  // 2 x TE
    uint64_t *full = reinterpret_cast<uint64_t *>(sums + 2 * G.te);
    uint64_t *empty = full + G.stages;
    auto red = reinterpret_cast<Stats<SCHEME>(*)[kBlock / 32]>(empty + G.stages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kOffset = SCHEME == kUniform;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) {
            mbar_init(&full[s], 1 + 32);           // producer's expect_tx + 32 cp.async arrivals
            mbar_init(&empty[s], kConsumerWarps);  // one arrival per consumer warp
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        bool ok = true;
        uint32_t it = 0;
        for (uint64_t tile = blockIdx.x; ok && tile < G.ntiles; tile += gridDim.x) {
            const uint64_t t0 = tile * G.te;
            const uint64_t tcnt = min(static_cast<uint64_t>(G.te), P.n - t0);
            const uint32_t wb = floor16((tcnt * BITS + 7u) / 8u);  // whole 16-byte units per worker
            const uint64_t k0 = tile * G.tb;
            for (uint32_t c = 0; c < G.nchunks; ++c, ++it) {
                const uint32_t s = it % G.stages;
                if (it >= G.stages && !mbar_wait(&empty[s], ((it / G.stages) - 1u) & 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t w0 = c * G.mc;
                const uint32_t mc = min(G.mc, static_cast<uint32_t>(P.M) - w0);
                unsigned char *stage = smem + s * G.stage_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[s], wb * mc);
                    if (wb)
                        for (uint32_t w = 0; w < mc; ++w)
                            bulk_load(stage + static_cast<size_t>(w) * G.worker_bytes,
                                      P.codes + (w0 + w) * P.codes_stride + (t0 * BITS) / 32u, wb,
                                      &full[s]);
                }
                float *msc = reinterpret_cast<float *>(stage + G.meta_offset);  // (scale, offset)
                for (uint32_t idx = lane; idx < mc * G.tb; idx += 32) {
                    const uint32_t w = idx / G.tb, kb = idx - w * G.tb;
                    if (k0 + kb < P.nbuckets) {
                        const uint64_t src = (w0 + w) * P.meta_stride + k0 + kb;
                        cp_async4(msc + 2 * idx, P.scale + src);
                        if constexpr (kOffset) cp_async4(msc + 2 * idx + 1, P.offset + src);
                    }
                }
                cp_async_arrive(&full[s]);
            }
        }
        cp_async_wait_all();
        if (!ok) {
            if (lane == 0) report_failure(&g_reencode_errors, P.status, kErrPipelineTimeout);
            // let copies already issued land (bounded)
            for (uint32_t d = 0; d < G.stages; ++d) {
                const uint32_t j = it >= G.stages ? it - G.stages + d : d;
                if (j < it) mbar_wait(&full[j % G.stages], (j / G.stages) & 1u);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ct = warp * 32 + lane;
    const float Mf = static_cast<float>(P.M);
    const int W = P.team_warps;
    const int teams = kConsumerWarps / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint32_t window = static_cast<uint32_t>(team_threads) * kSlots * 4u;
    int buf = 0;
    uint32_t it = 0, parity = 0;
    for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, parity ^= 1u) {
        const uint64_t t0 = tile * G.te;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(G.te), P.n - t0));
        const uint32_t wb = floor16((static_cast<uint64_t>(tcnt) * BITS + 7u) / 8u);
        const uint32_t *gcodes = P.codes + (t0 * BITS) / 32u;
        float *pb = sums + parity * G.te;
        bool ok = true;

        // ---- phase 1: decode and accumulate, chunk by chunk, into pb
        if (G.te == 16u * kConsumers && tcnt == G.te) {
            // One group of 16 consecutive outputs (all in one bucket) per
            // thread: the sums stay in registers across the chunks and pb is
            // written once.
            const uint32_t e = static_cast<uint32_t>(ct) * 16u;
            const uint32_t kb = G.bucket_shift >= 0 ? (e >> G.bucket_shift) : (e / P.bucket);
            float a[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) a[k] = 0.0f;
            float4 *ps = reinterpret_cast<float4 *>(pb + e);
            for (uint32_t c = 0; c < G.nchunks; ++c, ++it) {
                const uint32_t s = it % G.stages;
                if constexpr (EF) {
                    // the residual lands in this thread's own slots of pb (free
                    // until the end of the phase) while the last chunk runs
                    if (c + 1 == G.nchunks) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            cp_async16(ps + q4, reinterpret_cast<const float4 *>(P.err + t0 + e) + q4);
                    }
                }
                if (ok) ok = mbar_wait(&full[s], (it / G.stages) & 1u);
                if (ok) {
                    const unsigned char *stage = smem + s * G.stage_bytes;
                    const float2 *meta = reinterpret_cast<const float2 *>(stage + G.meta_offset) + kb;
                    const int mc = static_cast<int>(min(G.mc, static_cast<uint32_t>(P.M) - c * G.mc));
                    const unsigned char *wst = stage + (e * BITS) / 8u;
#pragma unroll 4
                    for (int w = 0; w < mc; ++w) {
                        uint32_t f[4];
                        load_codes16<BITS>(wst, f);
                        const float2 m = meta[w * G.tb];
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            a[k] = accumulate16<SCHEME, BITS>(a[k], f, k, m.x, m.y);
                        wst += G.worker_bytes;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if constexpr (EF) cp_async_wait_all();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float4 v = make_float4(finish_r(a[4 * q4], P, Mf), finish_r(a[4 * q4 + 1], P, Mf),
                                       finish_r(a[4 * q4 + 2], P, Mf), finish_r(a[4 * q4 + 3], P, Mf));
                if (P.out) __stcs(reinterpret_cast<float4 *>(P.out + t0 + e) + q4, v);
                if constexpr (EF) {
                    const float4 ev = ps[q4];
                    v = make_float4(__fadd_rn(ev.x, v.x), __fadd_rn(ev.y, v.y), __fadd_rn(ev.z, v.z),
                                    __fadd_rn(ev.w, v.w));
                }
                ps[q4] = v;
            }
        } else
        for (uint32_t c = 0; c < G.nchunks; ++c, ++it) {
            const uint32_t s = it % G.stages;
            if (ok) ok = mbar_wait(&full[s], (it / G.stages) & 1u);
            if (ok) {
                const unsigned char *stage = smem + s * G.stage_bytes;
                const float2 *msc = reinterpret_cast<const float2 *>(stage + G.meta_offset);
                const uint32_t w0 = c * G.mc;
                const int mc = static_cast<int>(min(G.mc, static_cast<uint32_t>(P.M) - w0));
                const bool first = c == 0, last = c + 1 == G.nchunks;
                if (tcnt == G.te) {
                    // 16 consecutive outputs per thread, all in one bucket.
                    for (uint32_t g = static_cast<uint32_t>(ct); g < G.te / 16u; g += kConsumers) {
                        const uint32_t e = g * 16u;
                        const uint32_t kb = G.bucket_shift >= 0 ? (e >> G.bucket_shift) : (e / P.bucket);
                        float a[16];
                        float4 *ps = reinterpret_cast<float4 *>(pb + e);
                        float4 ev[4];  // the residual, in flight during the worker loop
                        if constexpr (EF) {
                            if (last) {
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4)
                                    ev[q4] = __ldcs(reinterpret_cast<const float4 *>(P.err + t0 + e) + q4);
                            }
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float4 v = first ? make_float4(0.f, 0.f, 0.f, 0.f) : ps[q4];
                            a[4 * q4] = v.x; a[4 * q4 + 1] = v.y; a[4 * q4 + 2] = v.z; a[4 * q4 + 3] = v.w;
                        }
                        const unsigned char *wst = stage + (e * BITS) / 8u;
                        const float2 *meta = msc + kb;
#pragma unroll 4
                        for (int w = 0; w < mc; ++w) {
                            uint32_t f[4];
                            load_codes16<BITS>(wst, f);
                            const float2 m = meta[w * G.tb];
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                a[k] = accumulate16<SCHEME, BITS>(a[k], f, k, m.x, m.y);
                            wst += G.worker_bytes;
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            float4 v = make_float4(a[4 * q4], a[4 * q4 + 1], a[4 * q4 + 2], a[4 * q4 + 3]);
                            if (last) {
                                v = make_float4(finish_r(v.x, P, Mf), finish_r(v.y, P, Mf),
                                                finish_r(v.z, P, Mf), finish_r(v.w, P, Mf));
                                if (P.out) __stcs(reinterpret_cast<float4 *>(P.out + t0 + e) + q4, v);
                                if constexpr (EF) {
                                    v = make_float4(__fadd_rn(ev[q4].x, v.x), __fadd_rn(ev[q4].y, v.y),
                                                    __fadd_rn(ev[q4].z, v.z), __fadd_rn(ev[q4].w, v.w));
                                }
                            }
                            ps[q4] = v;
                        }
                    }
                } else {
                    // Tail tile: 4 outputs per thread; bytes past the staged
                    // part come from global memory.
                    for (uint32_t e = static_cast<uint32_t>(ct) * 4u; e < tcnt; e += kConsumers * 4u) {
                        const uint32_t kb = G.bucket_shift >= 0 ? (e >> G.bucket_shift) : (e / P.bucket);
                        const float2 *meta = msc + kb;
                        float a[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) a[k] = first ? 0.0f : pb[e + k];
                        for (int w = 0; w < mc; ++w) {
                            const uint32_t f = field4<BITS>(stage + static_cast<size_t>(w) * G.worker_bytes,
                                                            gcodes + (w0 + w) * P.codes_stride, e, wb);
                            const float2 m = meta[w * G.tb];
#pragma unroll
                            for (int k = 0; k < 4; ++k) a[k] = accumulate_code<SCHEME, BITS>(a[k], f, k, m.x, m.y);
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (e + k < tcnt) {
                                float v = a[k];
                                if (last) {
                                    v = finish_r(v, P, Mf);
                                    if (P.out) P.out[t0 + e + k] = v;
                                    if constexpr (EF) v = __fadd_rn(P.err[t0 + e + k], v);
                                }
                                pb[e + k] = v;
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---- phase 2: every consumer agrees the tile's sums are complete
        if (!consumer_sync_and<kConsumers>(ok)) {
            if (ct == 0) report_failure(&g_reencode_errors, P.status, kErrPipelineTimeout);
            break;
        }
        for (uint32_t kb0 = 0; kb0 < G.tb; kb0 += teams) {
            const uint32_t kb = kb0 + team;
            const uint32_t b_off = kb * P.bucket;
            const uint32_t cnt = (kb < G.tb && b_off < tcnt) ? min(P.bucket, tcnt - b_off) : 0u;
            // a bucket exactly one team window long takes the path without
            // per-slot bounds checks (uniform across the team)
            const bool whole = cnt == window;
            float4 p[kSlots];
            Stats<SCHEME> st;
            st.init();
            if (whole) {
                load_slots_sum<true>(pb, b_off, window, tt, team_threads, p);
                accumulate_slots<SCHEME, true>(st, p, tt, team_threads, window);
            } else {
                load_slots_sum(pb, b_off, min(cnt, window), tt, team_threads, p);
                accumulate_slots<SCHEME>(st, p, tt, team_threads, min(cnt, window));
                for (uint32_t w0 = window; w0 < cnt; w0 += window) {  // buckets above one window
                    float4 q[kSlots];
                    load_slots_sum(pb, b_off + w0, min(cnt - w0, window), tt, team_threads, q);
                    accumulate_slots<SCHEME>(st, q, tt, team_threads, min(cnt - w0, window));
                }
            }
            team_reduce<SCHEME, true>(st, red, buf, W, warp, lane, team);
            BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);
            if constexpr (SCHEME == kQsgd) {
                if (bp.exact) {  // rare: the norm next to a rounding boundary (uniform per team)
                    WideSum acc;
                    wide_zero(acc);
                    wide_add_slots(acc, p, tt, team_threads, min(cnt, window));
                    for (uint32_t w0 = window; w0 < cnt; w0 += window) {
                        float4 q[kSlots];
                        load_slots_sum(pb, b_off + w0, min(cnt - w0, window), tt, team_threads, q);
                        wide_add_slots(acc, q, tt, team_threads, min(cnt - w0, window));
                    }
                    // named barriers 8.. (barrier 1 belongs to the consumer group)
                    bp = qsgd_params<BITS>(team_exact_norm<SCHEME, 8>(acc, red, W, warp, lane, team));
                }
            }
            if (whole)
                quantize_store_slots<SCHEME, BITS, SR, EF, true>(P.codes_out, P.err, t0 + b_off, window,
                                                                 tt, team_threads, lane, p, bp, P.step,
                                                                 P.keys);
            else
                quantize_store_slots<SCHEME, BITS, SR, EF>(P.codes_out, P.err, t0 + b_off,
                                                           min(cnt, window), tt, team_threads, lane,
                                                           p, bp, P.step, P.keys);
            for (uint32_t w0 = window; w0 < cnt; w0 += window) {
                load_slots_sum(pb, b_off + w0, min(cnt - w0, window), tt, team_threads, p);
                quantize_store_slots<SCHEME, BITS, SR, EF>(P.codes_out, P.err, t0 + b_off + w0,
                                                           min(cnt - w0, window), tt, team_threads,
                                                           lane, p, bp, P.step, P.keys);
            }
            if (cnt && tt == 0) store_meta<SCHEME>(P.scale_out, P.offset_out, tile * G.tb + kb, bp);
        }
        // The other sum buffer takes the next tile, so no barrier is needed here:
        // this one is written again only after the next tile's agreement point.
    }
}

template <int SCHEME, int BITS, bool SR, bool EF>
cudaError_t launch_one(const ReencodeParams &p, const ReencodeTiles &g, cudaStream_t stream) {
    auto fn = &reencode_kernel<SCHEME, BITS, SR, EF>;
    const size_t smem = reencode_tiles_smem(g, sizeof(Stats<SCHEME>));
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kReBlock, g.ntiles, smem);
    fn<<<grid, kReBlock, smem, stream>>>(p, g);
    return cudaGetLastError();
}

template <int SCHEME, int BITS, bool SR>
cudaError_t launch_ef(const ReencodeParams &p, const ReencodeTiles &g, cudaStream_t stream) {
    return p.err ? launch_one<SCHEME, BITS, SR, true>(p, g, stream)
                 : launch_one<SCHEME, BITS, SR, false>(p, g, stream);
}

template <int SCHEME, int BITS>
cudaError_t launch_round(const ReencodeParams &p, const ReencodeTiles &g, int stochastic,
                         cudaStream_t stream) {
    return stochastic ? launch_ef<SCHEME, BITS, true>(p, g, stream)
                      : launch_ef<SCHEME, BITS, false>(p, g, stream);
}

}  // namespace
}  // namespace qc
