// qc_encode_bf16.cu -- encode of a bf16 gradient without error feedback (the
// receiver-side workload of a quantized all-reduce), streamed through the TMA
// shared-memory pipeline with 8 elements per lane slot.
//
// "Quantization for Communication", "Quantization Schemes" and "Quantized SGD
// Algorithms" (the arithmetic is the shared code in qc_encode_math.cuh);
// "Gradient Compression and Quantised Collectives", "When it breaks": gradients
// are already bf16 in a modern run.
//
// Without error feedback p = g exactly, so the bucket's min / max (uniform) or
// max |p| (ternary) are taken on packed bf16 pairs (one min.bf16x2 and one
// max.bf16x2 per two elements), and widened once at the end.  Lane slot s of
// team thread tt holds elements (s * 32 W + tt) * 8 .. +7 as one 16-byte
// shared-memory read; a team of W = ceil(bucket / 1024) warps owns a bucket, so
// the common bucket of 1024 needs no block barrier at all.
//
// Nor does the pipeline: each warp counts itself off a stage when it is done
// with it (a shared-memory counter), and the warp that completes the count
// refills the stage with the block's next tile but `stages`.  Warps therefore
// run up to two tiles apart instead of meeting at a barrier every tile.
#include "qc_encode_math.cuh"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_encode_bf16_errors;

namespace {

constexpr int kEps = 8;                       // elements per lane slot

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void unpack8(const uint4 &w, float (&v)[8]) {
    v[0] = __uint_as_float(w.x << 16);
    v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16);
    v[3] = __uint_as_float(w.y & 0xFFFF0000u);
    v[4] = __uint_as_float(w.z << 16);
    v[5] = __uint_as_float(w.z & 0xFFFF0000u);
    v[6] = __uint_as_float(w.w << 16);
    v[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// Packed statistics of full slots (bf16 pairs); partial slots go element-wise.
template <int SCHEME>
struct PackedStats {
    uint32_t a, b;
    __device__ void init() {
        if constexpr (SCHEME == kUniform) {
            a = 0x7F807F80u;  // +inf, +inf (running min)
            b = 0xFF80FF80u;  // -inf, -inf (running max)
        } else {
            a = 0u;  // running max |p|
            b = 0u;
        }
    }
    __device__ void add(uint32_t w) {
        if constexpr (SCHEME == kUniform) {
            a = bf16x2_min(a, w);
            b = bf16x2_max(b, w);
        } else {
            a = bf16x2_max(a, w & 0x7FFF7FFFu);
        }
    }
    __device__ void fold_into(Stats<SCHEME> &st) const {
        if constexpr (SCHEME == kUniform) {
            st.mn = fminf(st.mn, fminf(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u)));
            st.mx = fmaxf(st.mx, fmaxf(__uint_as_float(b << 16), __uint_as_float(b & 0xFFFF0000u)));
        } else if constexpr (SCHEME == kTernary || SCHEME == kLog) {  // max |p|
            st.add(__uint_as_float(a << 16));
            st.add(__uint_as_float(a & 0xFFFF0000u));
        }
    }
};

// Packs the 8 codes of a lane slot (c0 lowest) and stores them; every lane of
// the warp calls this together.
// `second`: the slot's last four elements exist (8-bit codes: their word is
// written only then; the other widths never start a word past the end).
template <int BITS>
__device__ __forceinline__ void store_codes8(uint32_t *codes, uint64_t i0, bool valid, int lane,
                                             uint32_t lo, uint32_t hi, bool second = true) {
    if constexpr (BITS == 8) {
        if (valid && second) __stcs(reinterpret_cast<uint2 *>(codes + i0 / 4u), make_uint2(lo, hi));
        else if (valid) __stcs(codes + i0 / 4u, lo);
    } else if constexpr (BITS == 4) {
        if (valid) __stcs(codes + i0 / 8u, lo | (hi << 16));
    } else if constexpr (BITS == 2) {
        uint32_t f = lo | (hi << 8);
        f |= __shfl_down_sync(kFull, f, 1) << 16;
        if (valid && (lane & 1) == 0) __stcs(codes + i0 / 16u, f);
    } else {
        uint32_t f = lo | (hi << 4);
        f |= __shfl_down_sync(kFull, f, 1) << 8;
        f |= __shfl_down_sync(kFull, f, 2) << 16;
        if (valid && (lane & 3) == 0) __stcs(codes + i0 / 32u, f);
    }
}

__device__ __forceinline__ void issue_tile(const EncodeParams &P, const EncodeTiles &G,
                                           uint64_t tile, unsigned char *stage, uint64_t *bar) {
    const uint64_t t0 = tile * G.te;
    const uint64_t tcnt = min(static_cast<uint64_t>(G.te), P.n - t0);
    const uint32_t gb = floor16(tcnt * 2u);
    mbar_arrive_expect_tx(bar, gb);
    if (gb) bulk_load(stage, static_cast<const uint16_t *>(P.grad) + t0, gb, bar);
}

// Stochastic ternary codes of the 8 elements of a slot, packed (element c in bits
// 2c, 2c+1), without conversions or selects: most of the work moves from the
// integer/logic pipe to the multiply-add pipe.
//   pa1 = fl(|v| * (1/s) + 1)          one fma
//   f   = 1 + (w >> 9) * 2^-23          the draw's top 23 bits as a mantissa
//   d   = f - pa1                       exact (both in [1, 2])
// d differs from u - fl(|v| / s) by less than 2^-22 (the reciprocal, the fma's
// rounding, the dropped 24th bit of u), so keep = [d < 0] is the exact decision
// whenever |d| > 2^-21; otherwise `near` is set and the caller recomputes the
// slot exactly.  Code bits: b0 = !keep, b1 = keep & (v >= +0).
__device__ __forceinline__ uint32_t ternary_sr_field8(const float (&v)[8], const uint4 &r0,
                                                      const uint4 &r1, float rinv, float delta2,
                                                      bool &near) {
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    uint32_t field = 0u, far = 0xFFFFFFFFu, m[8];
#pragma unroll
    for (int c = 7; c >= 0; --c) {
        const float pa1 = __fmaf_rn(fabsf(v[c]), rinv, 1.0f);
        // (0x7F : w) >> 9 = 0x3F800000 | (w >> 9): one funnel shift
        const float f = __uint_as_float(__funnelshift_r(w[c], 0x7Fu, 9));
        const float d = __fsub_rn(f, pa1);
        m[c] = __float_as_uint(__fsub_rn(delta2, fabsf(d)));  // sign set while |d| > delta2
        const uint32_t D = __float_as_uint(d);
        const uint32_t x = D & ~__float_as_uint(v[c]);
        field = __funnelshift_l(x, field, 1);   // b1 = keep & !sign(v)
        field = __funnelshift_l(D, field, 1);   // keep, inverted below
    }
#pragma unroll
    for (int c = 0; c < 8; c += 2) far &= m[c] & m[c + 1];
    near = (far >> 31) == 0u;
    return field ^ 0x5555u;
}

// 8-bit nearest codes of the 8 elements of a slot, four per word.  y = ta +
// 1.5 * 2^23 holds rint(ta) in its low mantissa bits and ta <= 255 (1 + 2^-22),
// so the low byte of y's bit pattern is the code itself: three byte permutes
// pack four codes.  `near` is set when some ta lies within reach of a
// half-integer (the caller recomputes those elements with the division).
__device__ __forceinline__ void uniform8_rn_fields(const float (&v)[8], const BucketParams &bp,
                                                   const FastQ &fq, uint32_t &f0, uint32_t &f1,
                                                   bool &near) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const float thr = 0.5f - fq.delta2;
    uint32_t y[8];
    bool any = false;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float ta = __fmul_rn(__fsub_rn(v[c], bp.a), fq.rinv);
        const float yf = __fadd_rn(ta, kMagic);
        y[c] = __float_as_uint(yf);
        any |= fabsf(__fsub_rn(ta, __fsub_rn(yf, kMagic))) >= thr;
    }
    f0 = __byte_perm(__byte_perm(y[0], y[1], 0x0040), __byte_perm(y[2], y[3], 0x0040), 0x5410);
    f1 = __byte_perm(__byte_perm(y[4], y[5], 0x0040), __byte_perm(y[6], y[7], 0x0040), 0x5410);
    near = any;
}

template <int SCHEME, int BITS, bool SR>
__global__ void __launch_bounds__(kBlock, 4) encode_bf16_kernel(const __grid_constant__ EncodeParams P,
                                                             const __grid_constant__ EncodeTiles G) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G.stages * G.stage_bytes);
    auto red = reinterpret_cast<Stats<SCHEME>(*)[kBlock / 32]>(full + G.stages);
    // per stage: warps done with its current tile (cumulative), and tiles issued into it
    uint32_t *done = reinterpret_cast<uint32_t *>(red + 2);
    uint32_t *issued = done + G.stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = G.warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const int team_threads = W * 32;
    const uint16_t *gsrc = static_cast<const uint16_t *>(P.grad);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0u;
            issued[s] = 0u;
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < G.stages; ++s) {
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(s) * gridDim.x;
            if (tile < G.ntiles) {
                issue_tile(P, G, tile, smem + s * G.stage_bytes, &full[s]);
                issued[s] = 1u;
            }
        }
    }
    const PhiloxKeys &keys = P.keys;

    int buf = 0;
    uint32_t it = 0;
    bool failed = false;
    for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % G.stages;
        const uint32_t parity = (it / G.stages) & 1u;
        const unsigned char *stage = smem + s * G.stage_bytes;
        // the team agrees on the wait's outcome, so its shuffles and barriers stay whole
        if (!team_all(mbar_wait(&full[s], parity), W, team)) {
            failed = true;
            break;
        }

        const uint64_t t0 = tile * G.te;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(G.te), P.n - t0));
        const uint32_t staged = floor16(static_cast<uint64_t>(tcnt) * 2u) / 2u;
        for (uint32_t kb0 = 0; kb0 < G.tb; kb0 += teams) {
            const uint32_t kb = kb0 + team;
            const uint32_t b_off = kb * P.bucket;
            const uint32_t cnt = (kb < G.tb && b_off < tcnt) ? min(P.bucket, tcnt - b_off) : 0u;
            const uint64_t b0 = t0 + b_off;

            // ---- load the lane's slots and take the statistics
            uint4 raw[kSlots];
            Stats<SCHEME> st;
            st.init();
            PackedStats<SCHEME> ps;
            ps.init();
            // QSGD: each pair of slots (16 elements) is summed into a fresh double
            // word and merged (the bound in Stats<kQsgd> counts 16 per window)
            Stats<SCHEME> part;
            part.init();
            Stats<SCHEME> &acc = (SCHEME == kQsgd) ? part : st;
#pragma unroll
            for (int sl = 0; sl < kSlots; ++sl) {
                const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * kEps;
                const uint32_t e = b_off + j;
                raw[sl] = make_uint4(0u, 0u, 0u, 0u);
                if (j + kEps <= cnt && e + kEps <= staged) {
                    raw[sl] = *reinterpret_cast<const uint4 *>(stage + e * 2u);
                    if constexpr (SCHEME == kSign || SCHEME == kQsgd) {
                        float v[8];
                        unpack8(raw[sl], v);
#pragma unroll
                        for (int c = 0; c < kEps; ++c) acc.add(v[c]);
                    } else {
                        ps.add(raw[sl].x);
                        ps.add(raw[sl].y);
                        ps.add(raw[sl].z);
                        ps.add(raw[sl].w);
                    }
                } else if (j < cnt) {  // ragged end: element-wise, from smem or global
                    uint32_t h[kEps];
#pragma unroll
                    for (int c = 0; c < kEps; ++c) {
                        h[c] = 0u;
                        if (j + c < cnt) {
                            h[c] = (e + c < staged)
                                       ? *reinterpret_cast<const unsigned short *>(stage + (e + c) * 2u)
                                       : __ldcs(reinterpret_cast<const unsigned short *>(gsrc + t0 + e + c));
                            acc.add(bf16_bits_to_float(h[c]));
                        }
                    }
                    raw[sl] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                         h[4] | (h[5] << 16), h[6] | (h[7] << 16));
                }
                if constexpr (SCHEME == kQsgd) {
                    if (sl & 1) {
                        st.merge(part);
                        part.init();
                    }
                }
            }
            ps.fold_into(st);
            team_reduce_local<SCHEME>(st, red, buf, W, warp, lane, team);
            BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);
            if constexpr (SCHEME == kQsgd) {
                if (bp.exact) {  // rare: the norm next to a rounding boundary (uniform per team)
                    WideSum wacc;
                    wide_zero(wacc);
#pragma unroll
                    for (int sl = 0; sl < kSlots; ++sl) {
                        const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * kEps;
                        const uint32_t w8[4] = {raw[sl].x, raw[sl].y, raw[sl].z, raw[sl].w};
#pragma unroll
                        for (int c = 0; c < kEps; ++c)
                            if (j + c < cnt)
                                wide_add_square(wacc, bf16_bits_to_float((w8[c >> 1] >> ((c & 1) * 16)) & 0xFFFFu));
                    }
                    bp = qsgd_params<BITS>(team_exact_norm<SCHEME, 1>(wacc, red, W, warp, lane, team));
                }
            }
            const FastQ fq = fast_params<SCHEME, BITS>(bp);

            // ---- quantize, pack and store, one slot at a time: a division-free
            // pass, an exact recompute of the slot in the rare case that one of its
            // elements lies near a decision boundary, then the store
            // whole buckets take the fast path; the test is uniform across the
            // team, so the packing shuffles always see the whole warp
            const uint32_t window = static_cast<uint32_t>(team_threads) * kSlots * kEps;
            if (fq.usable && cnt == window && b_off + window <= staged) {
#pragma unroll 2
                for (int sl = 0; sl < kSlots; ++sl) {
                    const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * kEps;
                    const uint64_t i0 = b0 + j;
                    float v[8], u[8];
                    unpack8(*reinterpret_cast<const uint4 *>(stage + (b_off + j) * 2u), v);
                    if constexpr (SCHEME == kUniform && BITS == 8 && !SR) {
                        uint32_t f0, f1;
                        bool near;
                        uniform8_rn_fields(v, bp, fq, f0, f1, near);
                        if (near) {  // rare: recompute the flagged elements with the division
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                bool r;
                                (void)code_fast<SCHEME, BITS, SR>(v[c], 0.0f, bp, fq, r);
                                if (r) {
                                    const uint32_t q = code_exact<SCHEME, BITS, SR>(v[c], 0.0f, bp);
                                    const int sh = (c & 3) * 8;
                                    if (c < 4) f0 = (f0 & ~(0xFFu << sh)) | (q << sh);
                                    else f1 = (f1 & ~(0xFFu << sh)) | (q << sh);
                                }
                            }
                        }
                        store_codes8<BITS>(P.codes, i0, true, lane, f0, f1);
                    } else if constexpr (SCHEME == kTernary && SR) {
                        bool near;
                        const uint32_t f16 = ternary_sr_field8(v, philox_words(P.index_base + i0, P.step, keys),
                                                               philox_words(P.index_base + i0 + 4, P.step, keys),
                                                               fq.rinv, fq.delta2, near);
                        uint32_t f0 = f16 & 0xFFu, f1 = f16 >> 8;
                        if (near) {  // rare: recompute the slot with the division
                            uniform4(P.index_base + i0, P.step, keys, u);
                            uniform4(P.index_base + i0 + 4, P.step, keys, u + 4);
                            f0 = f1 = 0;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                f0 |= code_exact<SCHEME, BITS, SR>(v[c], u[c], bp) << (c * BITS);
                                f1 |= code_exact<SCHEME, BITS, SR>(v[c + 4], u[c + 4], bp) << (c * BITS);
                            }
                        }
                        store_codes8<BITS>(P.codes, i0, true, lane, f0, f1);
                    } else {
#pragma unroll
                        for (int c = 0; c < kEps; ++c) u[c] = 0.0f;
                        if constexpr (SR) {
                            uniform4(P.index_base + i0, P.step, keys, u);
                            uniform4(P.index_base + i0 + 4, P.step, keys, u + 4);
                        }
                        uint32_t f0 = 0, f1 = 0;
                        bool any = false;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            bool r0, r1;
                            f0 |= code_fast<SCHEME, BITS, SR>(v[c], u[c], bp, fq, r0) << (c * BITS);
                            f1 |= code_fast<SCHEME, BITS, SR>(v[c + 4], u[c + 4], bp, fq, r1) << (c * BITS);
                            any |= r0 | r1;
                        }
                        if constexpr (SCHEME == kUniform) {
                            // rare (bf16 gradients land exactly on a tie a few times in
                            // a thousand): find the flagged elements again and recompute
                            // only those with the division
                            if (any) {
                                constexpr uint32_t kMask = (1u << BITS) - 1u;
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    bool r;
                                    (void)code_fast<SCHEME, BITS, SR>(v[c], u[c], bp, fq, r);
                                    if (r) {
                                        const uint32_t q = code_exact<SCHEME, BITS, SR>(v[c], u[c], bp);
                                        const int sh = (c & 3) * BITS;
                                        if (c < 4) f0 = (f0 & ~(kMask << sh)) | (q << sh);
                                        else f1 = (f1 & ~(kMask << sh)) | (q << sh);
                                    }
                                }
                            }
                        } else if (any) {  // rare: recompute the whole slot
                            f0 = f1 = 0;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                f0 |= code_exact<SCHEME, BITS, SR>(v[c], u[c], bp) << (c * BITS);
                                f1 |= code_exact<SCHEME, BITS, SR>(v[c + 4], u[c + 4], bp) << (c * BITS);
                            }
                        }
                        store_codes8<BITS>(P.codes, i0, true, lane, f0, f1);
                    }
                }
            } else {  // partial slots or an extreme scale: element-wise with the division
#pragma unroll
                for (int sl = 0; sl < kSlots; ++sl) {
                    const uint32_t j = static_cast<uint32_t>(sl * team_threads + tt) * kEps;
                    float v[8], u[8];
                    unpack8(raw[sl], v);
#pragma unroll
                    for (int c = 0; c < kEps; ++c) u[c] = 0.0f;
                    if constexpr (SR) {
                        if (j < cnt) {
                            uniform4(P.index_base + b0 + j, P.step, keys, u);
                            uniform4(P.index_base + b0 + j + 4, P.step, keys, u + 4);
                        }
                    }
                    uint32_t f0 = 0, f1 = 0;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (j + c < cnt) f0 |= code_exact<SCHEME, BITS, SR>(v[c], u[c], bp) << (c * BITS);
                        if (j + c + 4 < cnt)
                            f1 |= code_exact<SCHEME, BITS, SR>(v[c + 4], u[c + 4], bp) << (c * BITS);
                    }
                    store_codes8<BITS>(P.codes, b0 + j, j < cnt, lane, f0, f1, j + 4 < cnt);
                }
            }
            if (cnt && tt == 0) store_meta<SCHEME>(P.scale, P.offset, tile * G.tb + kb, bp);
        }
        // this warp is done with the stage (its reads have returned: their values
        // are used above); the warp that completes the count refills the stage
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t before = atomicAdd(&done[s], 1u);
            if (before % (kBlock / 32) == (kBlock / 32) - 1) {
                __threadfence_block();
                fence_proxy_async_shared();  // generic reads before the bulk copy's writes
                const uint64_t next = tile + static_cast<uint64_t>(G.stages) * gridDim.x;
                if (next < G.ntiles) {
                    issue_tile(P, G, next, smem + s * G.stage_bytes, &full[s]);
                    issued[s] += 1u;
                }
            }
        }
    }
    if (failed && lane == 0) report_failure(&g_encode_bf16_errors, P.status, kErrPipelineTimeout);
    // A team that gave up leaves its stages unrefilled, so the other teams' waits
    // run out too; every warp gets here.  Copies still in flight (only after a
    // failure) must land before the block's shared memory goes away.
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t d = 0; d < G.stages; ++d)
            if (issued[d]) mbar_wait(&full[d], (issued[d] - 1u) & 1u);
    }
}

template <int SCHEME, int BITS, bool SR>
cudaError_t launch_one(const EncodeParams &p, const EncodeTiles &g, cudaStream_t stream) {
    auto fn = &encode_bf16_kernel<SCHEME, BITS, SR>;
    const size_t smem = encode_tiles_smem(g, sizeof(Stats<SCHEME>));
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kBlock, g.ntiles, smem);
    fn<<<grid, kBlock, smem, stream>>>(p, g);
    return cudaGetLastError();
}

template <int SCHEME, int BITS>
cudaError_t launch_round(const EncodeParams &p, const EncodeTiles &g, int stochastic,
                         cudaStream_t stream) {
    return stochastic ? launch_one<SCHEME, BITS, true>(p, g, stream)
                      : launch_one<SCHEME, BITS, false>(p, g, stream);
}

}  // namespace

cudaError_t launch_encode_bf16(const EncodeParams &p, const EncodeTiles &g, int scheme, int bits,
                               int stochastic, cudaStream_t stream) {
    if (scheme == kSign) return launch_one<kSign, 1, false>(p, g, stream);
    if (scheme == kTernary) return launch_round<kTernary, 2>(p, g, stochastic, stream);
    if (scheme == kQsgd) {
        if (bits == 2) return launch_round<kQsgd, 2>(p, g, stochastic, stream);
        if (bits == 4) return launch_round<kQsgd, 4>(p, g, stochastic, stream);
        return launch_round<kQsgd, 8>(p, g, stochastic, stream);
    }
    if (scheme == kLog) {
        if (bits == 2) return launch_round<kLog, 2>(p, g, stochastic, stream);
        if (bits == 4) return launch_round<kLog, 4>(p, g, stochastic, stream);
        return launch_round<kLog, 8>(p, g, stochastic, stream);
    }
    switch (bits) {
        case 1: return launch_round<kUniform, 1>(p, g, stochastic, stream);
        case 2: return launch_round<kUniform, 2>(p, g, stochastic, stream);
        case 4: return launch_round<kUniform, 4>(p, g, stochastic, stream);
        default: return launch_round<kUniform, 8>(p, g, stochastic, stream);
    }
}

QC_DEFINE_TAKE_FLAG(take_encode_bf16_errors, g_encode_bf16_errors)

}  // namespace qc
