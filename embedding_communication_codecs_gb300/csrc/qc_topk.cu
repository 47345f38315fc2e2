// qc_topk.cu -- top-k sparsification with 8-bit quantization of the kept
// values and error feedback, and its receiver.
//
// "Gradient quantization for communication", "Quantization Schemes" (Top-K
// Sparsification: send only the largest K% of gradients, combined with
// quantization; Error Feedback); "Quantization for Communication",
// "Combination with Other Techniques" (quantize the sparse gradients);
// "Gradient Compression and Quantised Collectives", "Why sparsification fights
// the all-reduce" (the kept coordinates travel as index-value pairs, and the
// receiver sums an all-gather of them).
//
// Encode, per bucket of B <= 4096 elements (K = min(keep, cnt)):
//   p = e + g; the K elements of largest |p| (ties to the lower index) are
//   kept, in ascending index order, as (global index, 8-bit code) slots; the
//   codes are the uniform 8-bit quantization over the kept values' own min and
//   max; e = p - deq for kept elements, e = p for the others; unused slots of a
//   short last bucket hold index 0xFFFFFFFF and code 0.
// The kernel is the pipelined encode's (qc_encode_tma.cuh) tile and team
// layout.  The K-th largest |p| comes from team_select (qc_encode_math.cuh) on
// the keys bits(p) << 1: |p|'s bit pattern without its sign, moved up one bit
// so that the top byte is the exponent (one binade per histogram bin;
// non-negative floats order like their bit patterns).  One team
// scan in index order of two packed counters (keys >= T, keys == T) then gives
// every element whether it is kept (all keys > T, and the first `need` ties)
// and its output slot.
//
// Decode: a warp per bucket accumulates the workers' pairs into its own
// shared-memory copy of the bucket's output, worker by worker with a warp
// barrier in between (a worker's indices within a bucket are distinct, so each
// step is race-free and the fixed worker order holds), then writes the dense
// result.
#include "qc_encode_tma.cuh"

namespace qc {

static __device__ unsigned int g_topk_errors;

namespace {

constexpr uint32_t kNoIndex = 0xFFFFFFFFu;
constexpr int kScanWords = kTopkScanWords;  // per team: one total per slot and warp
static_assert(kScanWords == kSlots * (kBlock / 32), "scan totals");

// Exclusive prefix, in index order, of the lane's per-slot values a[s] over the
// team (slot-major, then lane order), and the team total.  Values are packed
// counters that never carry between halves.
__device__ __forceinline__ void team_scan(const uint32_t (&a)[kSlots], int W, int team,
                                          int warp_in_team, int lane, uint32_t *tot,
                                          uint32_t (&excl)[kSlots], uint32_t &total) {
    uint32_t incl[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        incl[s] = a[s];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, incl[s], o);
            if (lane >= o) incl[s] += t;
        }
        if (lane == 31) tot[s * 8 + warp_in_team] = incl[s];
    }
    team_sync(W, team);
    uint32_t running = 0u;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        uint32_t slot_total = 0u, before = 0u;
        for (int w = 0; w < W; ++w) {
            const uint32_t v = tot[s * 8 + w];
            slot_total += v;
            before += w < warp_in_team ? v : 0u;
        }
        excl[s] = running + before + (incl[s] - a[s]);
        running += slot_total;
    }
    total = running;
}

// One bucket of the team (cnt > 0): selection, the counter scan, the kept
// values' statistics, codes, slots, residuals and metadata.  FULL: every slot
// of the team's window is valid.
template <bool EF, bool SR, bool FULL>
__device__ __forceinline__ void topk_bucket(const TopkParams &T, const float4 (&p)[kSlots],
                                            uint32_t cnt, uint64_t b0, uint64_t k, int tt,
                                            int team_threads, int W, int team, int warp, int lane,
                                            uint32_t *region, uint32_t *tot,
                                            Stats<kUniform> (*red)[kBlock / 32], int &buf,
                                            uint32_t &parity) {
    const EncodeParams &P = T.e;
    const uint32_t K = min(T.keep, cnt);
    uint32_t key[kSlots][4];
#pragma unroll
    for (int sl = 0; sl < kSlots; ++sl)
#pragma unroll
        for (int c = 0; c < 4; ++c) key[sl][c] = __float_as_uint(get(p[sl], c)) << 1;
    uint32_t thr, unused;
    team_select<1, FULL>(key, cnt, P.bucket, cnt - K, cnt - K, tt, team_threads, W, team, warp % W,
                         lane, region, parity, thr, unused);
    // counters in index order: keys >= thr (low half), keys == thr (high half);
    // and the statistics of the values with keys >= thr and with keys > thr
    uint32_t a[kSlots];
    Stats<kUniform> st_ge, st_gt;
    st_ge.init();
    st_gt.init();
#pragma unroll
    for (int sl = 0; sl < kSlots; ++sl) {
        a[sl] = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * 4u + c;
            if (FULL || j < cnt) {
                const uint32_t kk = key[sl][c];
                a[sl] += (kk >= thr ? 1u : 0u) + (kk == thr ? 0x10000u : 0u);
                if (kk >= thr) st_ge.add(get(p[sl], c));
                if (kk > thr) st_gt.add(get(p[sl], c));
            }
        }
    }
    uint32_t excl[kSlots], total;
    team_scan(a, W, team, warp % W, lane, tot, excl, total);
    const uint32_t ties = total >> 16;
    const uint32_t need = K - ((total & 0xFFFFu) - ties);  // ties to keep, >= 1
    Stats<kUniform> st;
    if (need == ties) {
        st = st_ge;  // every tie is kept
    } else {         // rare: the first `need` ties in index order
        st = st_gt;
#pragma unroll
        for (int sl = 0; sl < kSlots; ++sl) {
            uint32_t run = excl[sl];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * 4u + c;
                if (FULL || j < cnt) {
                    const uint32_t kk = key[sl][c];
                    if (kk == thr && (run >> 16) < need) st.add(get(p[sl], c));
                    run += (kk >= thr ? 1u : 0u) + (kk == thr ? 0x10000u : 0u);
                }
            }
        }
    }
    team_reduce_local<kUniform>(st, red, buf, W, warp, lane, team);
    const BucketParams bp = Finish<kUniform, 8>::run(st, K);
#pragma unroll
    for (int sl = 0; sl < kSlots; ++sl) {
        uint32_t run = excl[sl];
        float4 e = p[sl];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * 4u + c;
            if (FULL || j < cnt) {
                const uint32_t kk = key[sl][c];
                const uint32_t ge_before = run & 0xFFFFu, tie_before = run >> 16;
                if (kk > thr || (kk == thr && tie_before < need)) {
                    const uint64_t i = b0 + j;
                    float u = 0.0f;
                    if constexpr (SR) u = uniform1(i, P.step, P.keys);
                    float deq;
                    const uint32_t q = quantize<kUniform, 8, SR>(get(p[sl], c), u, bp, deq);
                    const uint32_t pos = (ge_before - tie_before) + min(tie_before, need);
                    T.idx[k * T.keep + pos] = static_cast<uint32_t>(i);
                    T.codes8[k * T.keep + pos] = static_cast<uint8_t>(q);
                    set(e, c, __fsub_rn(get(p[sl], c), deq));
                }
                run += (kk >= thr ? 1u : 0u) + (kk == thr ? 0x10000u : 0u);
            }
        }
        if constexpr (EF) {
            const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * 4u;
            if (FULL || j + 4u <= cnt) {
                __stcs(reinterpret_cast<float4 *>(P.err + b0 + j), e);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (j + c < cnt) P.err[b0 + j + c] = get(e, c);
            }
        }
    }
    for (uint32_t t = K + static_cast<uint32_t>(tt); t < T.keep; t += team_threads) {
        T.idx[k * T.keep + t] = kNoIndex;
        T.codes8[k * T.keep + t] = 0;
    }
    if (tt == 0) store_meta<kUniform>(P.scale, P.offset, k, bp);
}

template <typename TIn, bool EF, bool SR>
__global__ void __launch_bounds__(kBlock) topk_kernel(const __grid_constant__ TopkParams T,
                                                      const __grid_constant__ EncodeTiles G) {
    const EncodeParams &P = T.e;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G.stages * G.stage_bytes);
    auto red = reinterpret_cast<Stats<kUniform>(*)[kBlock / 32]>(full + G.stages);
    uint32_t *teamwords = reinterpret_cast<uint32_t *>(red + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint32_t window = static_cast<uint32_t>(team_threads) * kSlots * 4u;
    const int region_words = sel_region_words(P.bucket) + kScanWords;
    uint32_t *region = teamwords + team * region_words;
    uint32_t *tot = region + sel_region_words(P.bucket);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    for (int i = threadIdx.x; i < teams * region_words; i += kBlock) teamwords[i] = 0u;
    __syncthreads();
    // the whole gradient is one segment of the pipelined encode's tiling
    const EncodeSeg seg{P.grad, P.err, P.n, nullptr, P.scale, P.offset, 0, 0};
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) {
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(s) * gridDim.x;
            if (tile < G.ntiles) issue_seg_tile<TIn, EF>(seg, G, tile, smem + s * G.stage_bytes, &full[s]);
        }
    }

    int buf = 0;
    uint32_t parity = 0, it = 0;
    bool failed = false;
    for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % G.stages;
        const unsigned char *stage = smem + s * G.stage_bytes;
        // the block agrees on the wait's outcome before computing or storing
        // anything (the selection is the bound here, not this barrier)
        if (!__syncthreads_and(mbar_wait(&full[s], (it / G.stages) & 1u))) {
            failed = true;
            break;
        }
        const uint64_t t0 = tile * G.te;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(G.te), P.n - t0));
        const uint32_t staged = staged_elems<TIn, EF>(tcnt);
        for (uint32_t kb0 = 0; kb0 < G.tb; kb0 += teams) {
            const uint32_t kb = kb0 + team;
            const uint32_t b_off = kb * P.bucket;
            const uint32_t cnt = (kb < G.tb && b_off < tcnt) ? min(P.bucket, tcnt - b_off) : 0u;
            const uint64_t b0 = t0 + b_off;
            const uint64_t k = tile * G.tb + kb;
            float4 p[kSlots];
            if (cnt == window && b_off + cnt <= staged) {
                load_slots_staged<TIn, EF, true>(seg, G, stage, t0, b_off, cnt, staged, tt, team_threads, p);
                topk_bucket<EF, SR, true>(T, p, cnt, b0, k, tt, team_threads, W, team, warp, lane,
                                          region, tot, red, buf, parity);
            } else if (cnt) {
                load_slots_staged<TIn, EF>(seg, G, stage, t0, b_off, cnt, staged, tt, team_threads, p);
                topk_bucket<EF, SR, false>(T, p, cnt, b0, k, tt, team_threads, W, team, warp, lane,
                                           region, tot, red, buf, parity);
            }
        }
        __syncthreads();  // every thread is done with this stage before it is refilled
        if (threadIdx.x == 0) {
            const uint64_t next = tile + static_cast<uint64_t>(G.stages) * gridDim.x;
            if (next < G.ntiles) issue_seg_tile<TIn, EF>(seg, G, next, smem + s * G.stage_bytes, &full[s]);
        }
    }
    if (failed && threadIdx.x == 0) {
        report_failure(&g_topk_errors, T.e.status, kErrPipelineTimeout);
        for (uint32_t d = 0; d < G.stages; ++d) {
            const uint32_t j = it + d;
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
            if (tile < G.ntiles) mbar_wait(&full[j % G.stages], (j / G.stages) & 1u);
        }
    }
}

constexpr int kDecodeMaxWarps = 8;
constexpr int kDecodeBatch = 8;  // workers whose pairs a lane holds in registers at once

// Dequantized value of one kept code (the uniform 8-bit level q * s + o, one
// rounding).
__device__ __forceinline__ float topk_level(uint32_t q, float s, float o) {
    return __fmaf_rn(__fsub_rn(__uint_as_float(q | 0x4B000000u), 8388608.0f), s, o);
}

// The warp's dense output pass over its bucket: finish, store, and zero the
// accumulators for the warp's next bucket.  MEAN: 0 none, 1 times inv_m (M a
// power of two, exact), 2 divided by M; ACC: add into the output's old value.
template <int MEAN, bool ACC>
__device__ __forceinline__ float topk_finish(float r, float prev, const TopkDecodeParams &D, float Mf) {
    if constexpr (MEAN == 1) r = __fmul_rn(r, D.inv_m);
    if constexpr (MEAN == 2) r = __fdiv_rn(r, Mf);
    if constexpr (ACC) r = __fadd_rn(prev, r);
    return r;
}

template <int MEAN, bool ACC>
__device__ __forceinline__ void topk_write_bucket(const TopkDecodeParams &D, float *acc, uint64_t lo,
                                                  uint32_t cnt, int lane, float Mf, bool vec) {
    uint32_t j0 = 0;
    if (vec) {  // bucket and output rows 16-byte aligned
        for (uint32_t j = 4u * static_cast<uint32_t>(lane); j + 4u <= cnt; j += 128u) {
            float4 *a4 = reinterpret_cast<float4 *>(acc + j);
            const float4 v = *a4;
            *a4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 *o4 = reinterpret_cast<float4 *>(D.out + lo + j);
            float4 prev = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (ACC) prev = *o4;
            __stcs(o4, make_float4(topk_finish<MEAN, ACC>(v.x, prev.x, D, Mf),
                                   topk_finish<MEAN, ACC>(v.y, prev.y, D, Mf),
                                   topk_finish<MEAN, ACC>(v.z, prev.z, D, Mf),
                                   topk_finish<MEAN, ACC>(v.w, prev.w, D, Mf)));
        }
        j0 = cnt & ~3u;
    }
    for (uint32_t j = j0 + static_cast<uint32_t>(lane); j < cnt; j += 32u) {
        const float v = acc[j];
        acc[j] = 0.0f;
        float *o = D.out + lo + j;
        *o = topk_finish<MEAN, ACC>(v, ACC ? *o : 0.0f, D, Mf);
    }
}

// M <= kDecodeBatch and keep <= 32: a lane holds its pair of every worker, and
// lane w holds worker w's scale and offset; the warp loads the pairs and
// metadata of its next bucket before it adds and writes the current one, so a
// bucket's loads are in flight while the previous bucket is processed.
template <int MEAN, bool ACC>
__device__ __forceinline__ void topk_decode_prefetched(const TopkDecodeParams &D, float *acc, int lane,
                                                       uint64_t first, uint64_t stride, float Mf,
                                                       bool vec) {
    const bool mine = static_cast<uint32_t>(lane) < D.keep;
    auto fetch = [&](uint64_t k, uint32_t (&iv)[kDecodeBatch], uint32_t (&qv)[kDecodeBatch], float &sl,
                     float &ol) {
#pragma unroll
        for (int b = 0; b < kDecodeBatch; ++b) {
            iv[b] = kNoIndex;
            qv[b] = 0u;
            if (b < D.M && mine) {
                const uint64_t at = static_cast<uint64_t>(b) * D.pair_stride + k * D.keep + lane;
                iv[b] = __ldg(D.idx + at);
                qv[b] = __ldg(D.codes8 + at);
            }
        }
        sl = ol = 0.0f;
        if (lane < D.M) {
            const uint64_t m = static_cast<uint64_t>(lane) * D.meta_stride + k;
            sl = __ldg(D.scale + m);
            ol = __ldg(D.offset + m);
        }
    };
    uint32_t iv[kDecodeBatch], qv[kDecodeBatch];
    float sl = 0.0f, ol = 0.0f;
    if (first < D.nbuckets) fetch(first, iv, qv, sl, ol);
    for (uint64_t k = first; k < D.nbuckets; k += stride) {
        uint32_t in[kDecodeBatch], qn[kDecodeBatch];
        float sn = 0.0f, on = 0.0f;
#pragma unroll
        for (int b = 0; b < kDecodeBatch; ++b) {
            in[b] = kNoIndex;
            qn[b] = 0u;
        }
        if (k + stride < D.nbuckets) fetch(k + stride, in, qn, sn, on);
        const uint64_t lo = k * D.bucket;
        const uint32_t cnt = static_cast<uint32_t>(min(static_cast<uint64_t>(D.bucket), D.n - lo));
#pragma unroll
        for (int b = 0; b < kDecodeBatch; ++b) {
            if (b >= D.M) break;  // uniform across the warp
            const float s = __shfl_sync(kFull, sl, b), o = __shfl_sync(kFull, ol, b);
            if (iv[b] >= lo && iv[b] < lo + cnt) {
                float *a = acc + (iv[b] - lo);
                *a = __fadd_rn(*a, topk_level(qv[b], s, o));
            }
            __syncwarp();
        }
        topk_write_bucket<MEAN, ACC>(D, acc, lo, cnt, lane, Mf, vec);
        __syncwarp();
#pragma unroll
        for (int b = 0; b < kDecodeBatch; ++b) {
            iv[b] = in[b];
            qv[b] = qn[b];
        }
        sl = sn;
        ol = on;
    }
}

// One bucket per warp: the bucket's accumulators live in the warp's part of
// shared memory; workers are added in their fixed order, a lane per kept pair,
// with only a warp barrier between workers (a worker's indices within a bucket
// are distinct, so the lanes of one step never touch the same accumulator).
// With keep <= 32 a lane loads its pair of the next kDecodeBatch workers ahead
// of adding them, so the loads of a batch overlap.  Pairs outside the bucket
// (the sentinel included) are skipped.
template <int MEAN, bool ACC>
__global__ void __launch_bounds__(kDecodeMaxWarps * 32) topk_decode_kernel(const __grid_constant__ TopkDecodeParams D) {
    extern __shared__ float sacc[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    float *acc = sacc + static_cast<size_t>(warp) * D.bucket;
    const float Mf = static_cast<float>(D.M);
    const bool vec = (D.bucket & 3u) == 0u && (reinterpret_cast<uintptr_t>(D.out) & 15u) == 0u;
    for (uint32_t j = static_cast<uint32_t>(lane); j < D.bucket; j += 32u) acc[j] = 0.0f;
    __syncwarp();
    if (D.M <= kDecodeBatch && D.keep <= 32u) {
        topk_decode_prefetched<MEAN, ACC>(D, acc, lane, static_cast<uint64_t>(blockIdx.x) * wpb + warp,
                                          static_cast<uint64_t>(gridDim.x) * wpb, Mf, vec);
        return;
    }
    for (uint64_t k = static_cast<uint64_t>(blockIdx.x) * wpb + warp; k < D.nbuckets;
         k += static_cast<uint64_t>(gridDim.x) * wpb) {
        const uint64_t lo = k * D.bucket;
        const uint32_t cnt = static_cast<uint32_t>(min(static_cast<uint64_t>(D.bucket), D.n - lo));
        if (D.keep <= 32u) {
            const bool mine = static_cast<uint32_t>(lane) < D.keep;
            for (int w0 = 0; w0 < D.M; w0 += kDecodeBatch) {
                uint32_t iv[kDecodeBatch], qv[kDecodeBatch];
                float sv[kDecodeBatch], ov[kDecodeBatch];
#pragma unroll
                for (int b = 0; b < kDecodeBatch; ++b) {
                    const int w = w0 + b;
                    iv[b] = kNoIndex;
                    qv[b] = 0u;
                    sv[b] = ov[b] = 0.0f;
                    if (w < D.M) {
                        const uint64_t at = static_cast<uint64_t>(w) * D.pair_stride + k * D.keep + lane;
                        if (mine) {
                            iv[b] = __ldg(D.idx + at);
                            qv[b] = __ldg(D.codes8 + at);
                        }
                        const uint64_t m = static_cast<uint64_t>(w) * D.meta_stride + k;
                        sv[b] = __ldg(D.scale + m);
                        ov[b] = __ldg(D.offset + m);
                    }
                }
#pragma unroll
                for (int b = 0; b < kDecodeBatch; ++b) {
                    if (w0 + b >= D.M) break;  // uniform across the warp
                    if (iv[b] >= lo && iv[b] < lo + cnt) {
                        float *a = acc + (iv[b] - lo);
                        *a = __fadd_rn(*a, topk_level(qv[b], sv[b], ov[b]));
                    }
                    __syncwarp();
                }
            }
        } else {
            for (int w = 0; w < D.M; ++w) {
                const uint64_t base = static_cast<uint64_t>(w) * D.pair_stride + k * D.keep;
                const uint64_t m = static_cast<uint64_t>(w) * D.meta_stride + k;
                const float s = __ldg(D.scale + m), o = __ldg(D.offset + m);
                for (uint32_t t = static_cast<uint32_t>(lane); t < D.keep; t += 32u) {
                    const uint32_t i = __ldg(D.idx + base + t);
                    if (i >= lo && i < lo + cnt) {
                        float *a = acc + (i - lo);
                        *a = __fadd_rn(*a, topk_level(__ldg(D.codes8 + base + t), s, o));
                    }
                }
                __syncwarp();
            }
        }
        topk_write_bucket<MEAN, ACC>(D, acc, lo, cnt, lane, Mf, vec);
        __syncwarp();
    }
}

template <typename TIn, bool EF, bool SR>
cudaError_t launch_one(const TopkParams &p, const EncodeTiles &g, cudaStream_t stream) {
    auto fn = &topk_kernel<TIn, EF, SR>;
    const int teams = (kBlock / 32) / p.e.team_warps;
    const size_t smem = encode_tiles_smem(g, sizeof(Stats<kUniform>)) +
                        static_cast<size_t>(teams) * (sel_region_words(p.e.bucket) + kScanWords) * 4u;
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kBlock, g.ntiles, smem);
    fn<<<grid, kBlock, smem, stream>>>(p, g);
    return cudaGetLastError();
}

template <bool SR>
cudaError_t launch_dtype(const TopkParams &p, const EncodeTiles &g, int bf16, cudaStream_t stream) {
    const bool ef = p.e.err != nullptr;
    if (bf16) return ef ? launch_one<uint16_t, true, SR>(p, g, stream) : launch_one<uint16_t, false, SR>(p, g, stream);
    return ef ? launch_one<float, true, SR>(p, g, stream) : launch_one<float, false, SR>(p, g, stream);
}

}  // namespace

cudaError_t launch_topk_encode(const TopkParams &p, const EncodeTiles &g, int stochastic, int bf16,
                               cudaStream_t stream) {
    return stochastic ? launch_dtype<true>(p, g, bf16, stream) : launch_dtype<false>(p, g, bf16, stream);
}

namespace {

template <int MEAN, bool ACC>
cudaError_t launch_decode_flags(const TopkDecodeParams &p, cudaStream_t stream) {
    // a warp per bucket, as many warps per block as keep the block's
    // accumulators within 64 KB
    const uint64_t bucket_bytes = static_cast<uint64_t>(p.bucket) * 4u;
    uint64_t fit = 65536u / bucket_bytes;
    if (fit < 1) fit = 1;
    const int wpb = static_cast<int>(fit < kDecodeMaxWarps ? fit : kDecodeMaxWarps);
    const size_t smem = static_cast<size_t>(wpb) * bucket_bytes;
    auto fn = &topk_decode_kernel<MEAN, ACC>;
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const uint64_t blocks = (p.nbuckets + wpb - 1) / wpb;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), wpb * 32, blocks, smem);
    fn<<<grid, wpb * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

template <bool ACC>
cudaError_t launch_decode_acc(const TopkDecodeParams &p, cudaStream_t stream) {
    if (!(p.flags & 1)) return launch_decode_flags<0, ACC>(p, stream);
    return p.inv_m != 0.0f ? launch_decode_flags<1, ACC>(p, stream) : launch_decode_flags<2, ACC>(p, stream);
}

}  // namespace

cudaError_t launch_topk_decode(const TopkDecodeParams &p, cudaStream_t stream) {
    return (p.flags & 2) ? launch_decode_acc<true>(p, stream) : launch_decode_acc<false>(p, stream);
}

QC_DEFINE_TAKE_FLAG(take_topk_errors, g_topk_errors)

}  // namespace qc
