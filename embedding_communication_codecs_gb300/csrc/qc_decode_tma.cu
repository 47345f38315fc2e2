// qc_decode_tma.cu -- receiver half of the codec with the M workers' payloads
// streamed into shared memory by a producer warp (TMA bulk copies for the code
// words, 4-byte cp.async for the per-bucket scales and offsets), consumed by
// eight warps that dequantize and accumulate in the fixed worker order.
//
// "Quantization for Communication", "Quantization-Aware All-Reduce" (dequantize
// after the exchange, accumulate in higher precision); "Gradient quantization for
// communication", "How Gradient Quantization Works" (dequantize, then average or
// sum).  Per element: acc = +0; for w = 0 .. M-1: acc = fl(acc + d_w); then
// optionally fl(acc / M) and fl(out + r).
//
// Tile = TB whole buckets (TE elements); one stage holds, for every worker, the
// TE * b / 8 code bytes of the tile followed by the M x TB scales and offsets.
// Warp specialisation: warp 8 is the producer; warps 0-7 consume.  A stage is
// refilled only after all eight consumer warps have arrived on its "empty"
// barrier, so consumer warps never wait for one another.  Every wait is bounded
// and a timeout is recorded in a device flag.
#include "qc_decode_math.cuh"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_decode_errors;

namespace {

constexpr int kDecodeBlock = kProducerBlock;

// The ternary decode's exponent fields and biases (accumulate_ternary16), read
// into registers once per thread.  They sit in memory so that the compiler
// cannot fold them into the logic operations as immediates.
__constant__ uint32_t kTernaryExp[8] = {150u << 23, 148u << 23, 146u << 23, 144u << 23,
                                        142u << 23, 140u << 23, 138u << 23, 136u << 23};
__constant__ float kTernaryBias[8] = {-8388609.0f, -2097153.0f, -524289.0f, -131073.0f,
                                      -32769.0f,   -8193.0f,    -2049.0f,   -513.0f};

template <int SCHEME, int BITS>
__global__ void __launch_bounds__(kDecodeBlock, SCHEME == kTernary ? 3 : 2) decode_tma_kernel(const __grid_constant__ DecodeParams P,
                                                                  const __grid_constant__ DecodeTiles G) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G.stages * G.stage_bytes);
    uint64_t *empty = full + G.stages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool kOffset = SCHEME == kUniform;
    const uint32_t meta_per_tile = static_cast<uint32_t>(P.M) * G.tb;

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
        for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, ++it) {
            const uint32_t s = it % G.stages;
            if (it >= G.stages && !mbar_wait(&empty[s], ((it / G.stages) - 1u) & 1u)) {
                ok = false;
                break;
            }
            unsigned char *stage = smem + s * G.stage_bytes;
            const uint64_t t0 = tile * G.te;
            const uint64_t tcnt = min(static_cast<uint64_t>(G.te), P.n - t0);
            const uint32_t wb = floor16((tcnt * BITS + 7u) / 8u);  // whole 16-byte units per worker
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], wb * static_cast<uint32_t>(P.M));
                if (wb)
                    for (int w = 0; w < P.M; ++w)
                        bulk_load(stage + static_cast<size_t>(w) * G.worker_bytes,
                                  P.codes + w * P.codes_stride + (t0 * BITS) / 32u, wb, &full[s]);
            }
            float *msc = reinterpret_cast<float *>(stage + G.meta_offset);  // (scale, offset) pairs
            const uint64_t k0 = tile * G.tb;
            for (uint32_t idx = lane; idx < meta_per_tile; idx += 32) {
                const uint32_t w = idx / G.tb, kb = idx - w * G.tb;
                if (k0 + kb < P.nbuckets) {
                    cp_async4(msc + 2 * idx, P.scale + w * P.meta_stride + k0 + kb);
                    if constexpr (kOffset)
                        cp_async4(msc + 2 * idx + 1, P.offset + w * P.meta_stride + k0 + kb);
                }
            }
            cp_async_arrive(&full[s]);
        }
        cp_async_wait_all();
        if (!ok) {
            if (lane == 0) report_failure(&g_decode_errors, P.status, kErrPipelineTimeout);
            // let copies already issued land (bounded)
            for (uint32_t d = 0; d < G.stages; ++d) {
                const uint32_t j = it >= G.stages ? it - G.stages + d : d;
                const uint64_t tile = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
                if (j < it && tile < G.ntiles) mbar_wait(&full[j % G.stages], (j / G.stages) & 1u);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ct = warp * 32 + lane;
    const float Mf = static_cast<float>(P.M);
    uint32_t tex[8];
    unsigned long long tk2[4];
    if constexpr (SCHEME == kTernary) {
#pragma unroll
        for (int j = 0; j < 8; ++j) tex[j] = kTernaryExp[j];
#pragma unroll
        for (int i = 0; i < 4; ++i) tk2[i] = pack2(kTernaryBias[2 * i], kTernaryBias[2 * i + 1]);
    }
    uint32_t it = 0;
    for (uint64_t tile = blockIdx.x; tile < G.ntiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % G.stages;
        if (!mbar_wait(&full[s], (it / G.stages) & 1u)) {
            if (lane == 0) report_failure(&g_decode_errors, P.status, kErrPipelineTimeout);
            break;
        }
        const unsigned char *stage = smem + s * G.stage_bytes;
        const float *msc = reinterpret_cast<const float *>(stage + G.meta_offset);
        const uint64_t t0 = tile * G.te;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(G.te), P.n - t0));
        const uint32_t wb = floor16((static_cast<uint64_t>(tcnt) * BITS + 7u) / 8u);
        const uint32_t *gcodes = P.codes + (t0 * BITS) / 32u;

        if (tcnt == G.te) {
            // Whole tile: each thread takes 16 consecutive outputs, which lie in
            // one bucket (buckets are multiples of 32), so one wide load gives a
            // worker's 16 codes and one 8-byte load its (scale, offset).
            for (uint32_t g = static_cast<uint32_t>(ct); g < G.te / 16u; g += kConsumerWarps * 32) {
                const uint32_t e = g * 16u;
                const uint32_t kb = G.bucket_shift >= 0 ? (e >> G.bucket_shift) : (e / P.bucket);
                const float2 *meta = reinterpret_cast<const float2 *>(msc) + kb;
                const unsigned char *wst = stage + (e * BITS) / 8u;
                float a[16];
                if constexpr (SCHEME == kTernary) {
                    // eight packed pairs; one word holds a worker's 16 codes
                    unsigned long long a2[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) a2[c] = 0ull;  // +0, +0
#pragma unroll 4
                    for (int w = 0; w < P.M; ++w) {
                        const uint32_t f = *reinterpret_cast<const uint32_t *>(wst);
                        const float sw = meta[w * G.tb].x;
                        accumulate_ternary16(a2, f, pack2(sw, sw), tex, tk2);
                        wst += G.worker_bytes;
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) unpack2(a2[c], a[2 * c], a[2 * c + 1]);
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) a[c] = 0.0f;
#pragma unroll 4
                    for (int w = 0; w < P.M; ++w) {
                        uint32_t f[4];
                        load_codes16<BITS>(wst, f);
                        const float2 m = meta[w * G.tb];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            a[c] = accumulate16<SCHEME, BITS>(a[c], f, c, m.x, m.y);
                        wst += G.worker_bytes;
                    }
                }
                float4 *o = reinterpret_cast<float4 *>(P.out + t0 + e);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float4 r = make_float4(a[4 * q4], a[4 * q4 + 1], a[4 * q4 + 2], a[4 * q4 + 3]);
                    if (P.flags & 1)
                        r = P.inv_m != 0.0f
                                ? make_float4(__fmul_rn(r.x, P.inv_m), __fmul_rn(r.y, P.inv_m),
                                              __fmul_rn(r.z, P.inv_m), __fmul_rn(r.w, P.inv_m))
                                : make_float4(__fdiv_rn(r.x, Mf), __fdiv_rn(r.y, Mf),
                                              __fdiv_rn(r.z, Mf), __fdiv_rn(r.w, Mf));
                    if (P.flags & 2) {
                        const float4 prev = __ldcs(o + q4);
                        r = make_float4(__fadd_rn(prev.x, r.x), __fadd_rn(prev.y, r.y),
                                        __fadd_rn(prev.z, r.z), __fadd_rn(prev.w, r.w));
                    }
                    __stcs(o + q4, r);
                }
            }
        } else {
            // Tail tile: 4 outputs per thread, bytes past the staged part read
            // from global memory.
            for (uint32_t e = static_cast<uint32_t>(ct) * 4u; e < tcnt; e += kConsumerWarps * 32 * 4) {
                const uint32_t kb = G.bucket_shift >= 0 ? (e >> G.bucket_shift) : (e / P.bucket);
                const float2 *meta = reinterpret_cast<const float2 *>(msc) + kb;
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
                for (int w = 0; w < P.M; ++w) {
                    const uint32_t f = field4<BITS>(stage + static_cast<size_t>(w) * G.worker_bytes,
                                                    gcodes + w * P.codes_stride, e, wb);
                    const float2 m = meta[w * G.tb];
                    a0 = accumulate_code<SCHEME, BITS>(a0, f, 0, m.x, m.y);
                    a1 = accumulate_code<SCHEME, BITS>(a1, f, 1, m.x, m.y);
                    a2 = accumulate_code<SCHEME, BITS>(a2, f, 2, m.x, m.y);
                    a3 = accumulate_code<SCHEME, BITS>(a3, f, 3, m.x, m.y);
                }
                float4 r = make_float4(a0, a1, a2, a3);
                if (P.flags & 1)
                    r = P.inv_m != 0.0f
                            ? make_float4(__fmul_rn(r.x, P.inv_m), __fmul_rn(r.y, P.inv_m),
                                          __fmul_rn(r.z, P.inv_m), __fmul_rn(r.w, P.inv_m))
                            : make_float4(__fdiv_rn(r.x, Mf), __fdiv_rn(r.y, Mf), __fdiv_rn(r.z, Mf),
                                          __fdiv_rn(r.w, Mf));
                const uint64_t i = t0 + e;
                if (e + 4u <= tcnt) {
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
                        if (e + c < tcnt) {
                            float v = get(r, c);
                            if (P.flags & 2) v = __fadd_rn(P.out[i + c], v);
                            P.out[i + c] = v;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

template <int SCHEME, int BITS>
cudaError_t launch_one(const DecodeParams &p, const DecodeTiles &g, cudaStream_t stream) {
    auto fn = &decode_tma_kernel<SCHEME, BITS>;
    const size_t smem = decode_tiles_smem(g);
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kDecodeBlock, g.ntiles, smem);
    fn<<<grid, kDecodeBlock, smem, stream>>>(p, g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tma(const DecodeParams &p, const DecodeTiles &g, int scheme, int bits,
                              cudaStream_t stream) {
    if (scheme == kSign) return launch_one<kSign, 1>(p, g, stream);
    if (scheme == kTernary) return launch_one<kTernary, 2>(p, g, stream);
    if (scheme == kLog) {
        if (bits == 2) return launch_one<kLog, 2>(p, g, stream);
        if (bits == 4) return launch_one<kLog, 4>(p, g, stream);
        return launch_one<kLog, 8>(p, g, stream);
    }
    if (scheme == kQsgd) {
        if (bits == 2) return launch_one<kQsgd, 2>(p, g, stream);
        if (bits == 4) return launch_one<kQsgd, 4>(p, g, stream);
        return launch_one<kQsgd, 8>(p, g, stream);
    }
    switch (bits) {
        case 1: return launch_one<kUniform, 1>(p, g, stream);
        case 2: return launch_one<kUniform, 2>(p, g, stream);
        case 4: return launch_one<kUniform, 4>(p, g, stream);
        default: return launch_one<kUniform, 8>(p, g, stream);
    }
}

QC_DEFINE_TAKE_FLAG(take_decode_errors, g_decode_errors)

}  // namespace qc
