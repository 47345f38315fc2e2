// qc_fp8.cu -- FP32 -> FP8 (OCP E4M3) row-wise quantization of embedding lookup
// payloads and its inverse.
//
// "Quantized Communication for Distributed Training", sections "Numeric Example"
// (1,000,000 lookups x 128 values: 512 MB in FP32, 128 MB in FP8) and "Pinterest
// QComms Example" (payloads go FP32 -> FP8 before the collective); the receiver
// dequantizes ("Where Quantization Sits").
//
// Per row: a = max |x|, sc = a / 448 (448 is E4M3's largest finite value), code =
// e4m3(x / sc) with round-to-nearest-even and saturation.  The conversion is the
// hardware cvt.rn.satfinite.e4m3x2.f32 instruction; decoding uses
// cvt.rn.f16x2.e4m3x2 (exact) followed by an exact f16 -> f32 widening.
//
// Layout: for dim <= 128 each warp takes four rows per step, one per float4
// slot, lane l covering columns 4l .. 4l+3 (four independent warp reductions,
// four 512-byte loads in flight per warp); both directions load the warp's next
// four rows before they process the current ones.  For wider rows a team of W warps
// owns a row with up to 4 float4 slots per lane.
#include "qc_device.cuh"
#include "qc_internal.h"

namespace qc {
namespace {

// Two E4M3 codes in one 16-bit value: `lo` in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four codes (bytes of `w`, lowest first) -> four exact fp32 values.
__device__ __forceinline__ float4 e4m3x4_to_float4(uint32_t w) {
    uint32_t h01, h23;
    const unsigned short lo = static_cast<unsigned short>(w & 0xFFFFu);
    const unsigned short hi = static_cast<unsigned short>(w >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(lo));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(hi));
    float f0, f1, f2, f3;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f0) : "h"(static_cast<unsigned short>(h01 & 0xFFFFu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f1) : "h"(static_cast<unsigned short>(h01 >> 16)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f2) : "h"(static_cast<unsigned short>(h23 & 0xFFFFu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f3) : "h"(static_cast<unsigned short>(h23 >> 16)));
    return make_float4(f0, f1, f2, f3);
}

__device__ __forceinline__ uint32_t encode4(const float4 &v, float sc) {
    if (sc == 0.0f) return 0u;
    const float y0 = __fdiv_rn(v.x, sc), y1 = __fdiv_rn(v.y, sc);
    const float y2 = __fdiv_rn(v.z, sc), y3 = __fdiv_rn(v.w, sc);
    return e4m3x2(y0, y1) | (e4m3x2(y2, y3) << 16);
}

__device__ __forceinline__ float absmax4(const float4 &v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// max over the warp's lanes of m >= +0, NaN lanes left out (+0 when every lane
// is NaN), as the row maximum ignores NaN elements.  Non-negative floats order
// like their bit patterns, so one integer max reduction replaces the
// five-step shuffle tree.
__device__ __forceinline__ float warp_absmax(float m) {
    return __uint_as_float(__reduce_max_sync(kFull, m == m ? __float_as_uint(m) : 0u));
}

constexpr int kRowsPerWarp = kSlots;  // dim <= 128: one row per slot

__global__ void __launch_bounds__(kBlock) fp8_quant_narrow(const Fp8Params P) {
    const int lane = threadIdx.x & 31;
    const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (kBlock / 32);
    const uint64_t groups = (P.rows + kRowsPerWarp - 1) / kRowsPerWarp;
    const bool col_ok = static_cast<uint32_t>(lane) * 4u < P.dim;
    // the rows of the warp's next group are loaded before the current group is
    // reduced and converted, so loads stay in flight during the arithmetic
    auto load = [&](uint64_t g, float4 (&v)[kRowsPerWarp]) {
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) {
            const uint64_t r = g * kRowsPerWarp + s;
            v[s] = (g < groups && col_ok && r < P.rows)
                       ? __ldcs(reinterpret_cast<const float4 *>(P.x + r * P.dim) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    uint64_t g = static_cast<uint64_t>(blockIdx.x) * (kBlock / 32) + (threadIdx.x >> 5);
    float4 cur[kRowsPerWarp];
    load(g, cur);
    for (; g < groups; g += warps) {
        float4 nxt[kRowsPerWarp];
        load(g + warps, nxt);
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) {
            const uint64_t r = g * kRowsPerWarp + s;
            const float sc = __fdiv_rn(warp_absmax(absmax4(cur[s])), 448.0f);
            if (col_ok && r < P.rows) {
                __stcs(reinterpret_cast<uint32_t *>(P.codes + r * P.dim) + lane, encode4(cur[s], sc));
                if (lane == 0) P.row_scale[r] = sc;
            }
        }
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) cur[s] = nxt[s];
    }
}

__global__ void __launch_bounds__(kBlock) fp8_quant_wide(const Fp8Params P) {
    __shared__ float red[2][kBlock / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const uint64_t groups = (P.rows + teams - 1) / teams;
    int buf = 0;
    for (uint64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const uint64_t r = grp * teams + team;
        const bool row_ok = r < P.rows;
        float4 v[kSlots];
        float m = 0.0f;
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const uint32_t col = static_cast<uint32_t>(s * W * 32 + tt) * 4u;
            v[s] = (row_ok && col < P.dim)
                       ? __ldcs(reinterpret_cast<const float4 *>(P.x + r * P.dim + col))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
            m = fmaxf(m, absmax4(v[s]));
        }
        m = warp_absmax(m);
        if (W > 1) {
            if (lane == 0) red[buf][warp] = m;
            __syncthreads();
            m = red[buf][team * W];
            for (int w = 1; w < W; ++w) m = fmaxf(m, red[buf][team * W + w]);
            buf ^= 1;
        }
        const float sc = __fdiv_rn(positive_zero(m), 448.0f);
        if (row_ok) {
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                const uint32_t col = static_cast<uint32_t>(s * W * 32 + tt) * 4u;
                if (col < P.dim)
                    __stcs(reinterpret_cast<uint32_t *>(P.codes + r * P.dim + col), encode4(v[s], sc));
            }
            if (tt == 0) P.row_scale[r] = sc;
        }
    }
}

__global__ void __launch_bounds__(kBlock) fp8_dequant_narrow(const Fp8Params P) {
    const int lane = threadIdx.x & 31;
    const uint64_t warps = static_cast<uint64_t>(gridDim.x) * (kBlock / 32);
    const uint64_t groups = (P.rows + kRowsPerWarp - 1) / kRowsPerWarp;
    const bool col_ok = static_cast<uint32_t>(lane) * 4u < P.dim;
    // the code words and scales of the warp's next group are loaded before the
    // current group is converted and stored, so loads stay in flight
    auto load = [&](uint64_t g, uint32_t (&cw)[kRowsPerWarp], float (&sc)[kRowsPerWarp]) {
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) {
            const uint64_t r = g * kRowsPerWarp + s;
            const bool ok = g < groups && col_ok && r < P.rows;
            cw[s] = ok ? __ldcs(reinterpret_cast<const uint32_t *>(P.codes_in + r * P.dim) + lane) : 0u;
            sc[s] = ok ? __ldg(P.scale_in + r) : 0.0f;
        }
    };
    uint64_t g = static_cast<uint64_t>(blockIdx.x) * (kBlock / 32) + (threadIdx.x >> 5);
    uint32_t cw[kRowsPerWarp];
    float sc[kRowsPerWarp];
    load(g, cw, sc);
    for (; g < groups; g += warps) {
        uint32_t cn[kRowsPerWarp];
        float sn[kRowsPerWarp];
        load(g + warps, cn, sn);
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) {
            const uint64_t r = g * kRowsPerWarp + s;
            if (col_ok && r < P.rows) {
                const float4 f = e4m3x4_to_float4(cw[s]);
                __stcs(reinterpret_cast<float4 *>(P.out + r * P.dim) + lane,
                       make_float4(__fmul_rn(f.x, sc[s]), __fmul_rn(f.y, sc[s]),
                                   __fmul_rn(f.z, sc[s]), __fmul_rn(f.w, sc[s])));
            }
        }
#pragma unroll
        for (int s = 0; s < kRowsPerWarp; ++s) {
            cw[s] = cn[s];
            sc[s] = sn[s];
        }
    }
}

__global__ void __launch_bounds__(kBlock) fp8_dequant_wide(const Fp8Params P) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = P.team_warps;
    const int teams = (kBlock / 32) / W;
    const int team = warp / W;
    const int tt = (warp % W) * 32 + lane;
    const uint64_t groups = (P.rows + teams - 1) / teams;
    for (uint64_t grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const uint64_t r = grp * teams + team;
        if (r >= P.rows) continue;
        const float sc = __ldg(P.scale_in + r);
        uint32_t cw[kSlots];
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const uint32_t col = static_cast<uint32_t>(s * W * 32 + tt) * 4u;
            cw[s] = col < P.dim ? __ldcs(reinterpret_cast<const uint32_t *>(P.codes_in + r * P.dim + col)) : 0u;
        }
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const uint32_t col = static_cast<uint32_t>(s * W * 32 + tt) * 4u;
            if (col < P.dim) {
                const float4 f = e4m3x4_to_float4(cw[s]);
                __stcs(reinterpret_cast<float4 *>(P.out + r * P.dim + col),
                       make_float4(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc), __fmul_rn(f.z, sc),
                                   __fmul_rn(f.w, sc)));
            }
        }
    }
}

}  // namespace

cudaError_t launch_fp8_quant(const Fp8Params &p, cudaStream_t stream) {
    if (p.dim <= 128) {
        const uint64_t groups = (p.rows + kRowsPerWarp - 1) / kRowsPerWarp;
        const int grid = persistent_grid(reinterpret_cast<const void *>(&fp8_quant_narrow), kBlock,
                                         (groups + (kBlock / 32) - 1) / (kBlock / 32));
        fp8_quant_narrow<<<grid, kBlock, 0, stream>>>(p);
    } else {
        const int teams = (kBlock / 32) / p.team_warps;
        const int grid = persistent_grid(reinterpret_cast<const void *>(&fp8_quant_wide), kBlock,
                                         (p.rows + teams - 1) / teams);
        fp8_quant_wide<<<grid, kBlock, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_fp8_dequant(const Fp8Params &p, cudaStream_t stream) {
    if (p.dim <= 128) {
        const uint64_t groups = (p.rows + kRowsPerWarp - 1) / kRowsPerWarp;
        const int grid = persistent_grid(reinterpret_cast<const void *>(&fp8_dequant_narrow),
                                         kBlock, (groups + (kBlock / 32) - 1) / (kBlock / 32));
        fp8_dequant_narrow<<<grid, kBlock, 0, stream>>>(p);
    } else {
        const int teams = (kBlock / 32) / p.team_warps;
        const int grid = persistent_grid(reinterpret_cast<const void *>(&fp8_dequant_wide), kBlock,
                                         (p.rows + teams - 1) / teams);
        fp8_dequant_wide<<<grid, kBlock, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace qc
