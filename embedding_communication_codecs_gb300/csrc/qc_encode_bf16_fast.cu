// qc_encode_bf16_fast.cu -- the receiver's two bf16 encodes without error
// feedback, for buckets of 1024 elements: 8-bit uniform with round to nearest
// and TernGrad ternary with stochastic rounding ("Quantization for
// Communication", "Quantization Schemes" and "Quantized SGD Algorithms";
// "Gradient Compression and Quantised Collectives", "When it breaks": the
// gradients are bf16).  They compute exactly what the general bf16 kernel
// computes (and what the oracle computes), with fewer instructions per element:
//
//  * tiles of 16 buckets in 32 KB stages, two buckets per warp, so that the
//    tile's bookkeeping (wait, segment, counts, refill) is paid once for both;
//  * one warp per bucket and 32 elements per lane (four 16-byte shared-memory
//    reads), which the 8-bit kernel holds in registers between the statistics
//    and the codes and the ternary kernel reads again for the codes;
//  * the statistics on packed bf16 pairs: max |x| with one max.xorsign.abs per
//    pair (only the magnitude of the result is used), min and max with one
//    min / max each;
//  * bf16 values widened (or widened and offset) by the mixed-precision
//    add.f32.bf16 on the FMA pipes instead of shifts and masks on the ALU;
//  * Philox4x32-10 with the rounds that depend only on (seed, step) folded on
//    the host (PhiloxStep): 18 instead of 20 wide multiplies per call;
//  * the two ternary code bits of an element built from the signs of two
//    differences and shifted in with one funnel shift.
//
// The division-free decisions keep the exact fallback of the general kernels:
// in a lane slot of 8 elements with an element within reach of a decision
// boundary, the ternary kernel recomputes the slot and the 8-bit kernel the
// flagged elements with the IEEE division.  A bucket that is not whole
// (the last one of the array) is encoded from global memory by the same warp
// with the exact element-wise code.
#include "qc_encode_math.cuh"
#include "qc_pipeline.cuh"

namespace qc {

static __device__ unsigned int g_encode_bf16_fast_errors;

namespace {

constexpr uint32_t kB = 1024;                        // bucket
constexpr int kWarps = kBlock / 32;                  // warps per block
constexpr uint32_t kPerWarp = 2;                     // buckets per warp and tile
constexpr uint32_t kTile = kB * kWarps * kPerWarp;   // elements per tile
constexpr uint32_t kStageBytes = kTile * 2u;         // 32 KB of bf16

constexpr int kU8 = 0;       // 8-bit uniform, round to nearest
constexpr int kTern = 1;     // ternary, stochastic rounding

constexpr uint32_t kStages = 2;
constexpr size_t kSmem = kStages * kStageBytes + kStages * 8u + 2u * kStages * 4u;

// A 16-byte shared-memory load the compiler may not merge with an earlier one.
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return r;
}

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t min_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// fl(x - c) for the bf16 half H (0 low, 1 high) of w: the half widened exactly,
// one rounding.  With c = +0 the result is the half itself (x - 0 = x, -0 kept).
template <int H>
__device__ __forceinline__ float bf16_sub(uint32_t w, float c) {
    float r;
    if constexpr (H == 0)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tsub.rn.f32.bf16 %0, l, %2;\n\t}"
            : "=f"(r)
            : "r"(w), "f"(c));
    else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tsub.rn.f32.bf16 %0, h, %2;\n\t}"
            : "=f"(r)
            : "r"(w), "f"(c));
    return r;
}

// Rounds of Philox4x32-10 for counter (blk, 0, step, 0): round 0's product of the
// step and round 1's product of round 0's first word depend only on (seed,
// step), so the host folds them into four constants (philox_step below).
struct PhiloxStep {
    uint32_t b0;  // key b of round 0
    uint32_t k1;  // lo(B * step) ^ a[1]                 (round 1, word 0)
    uint32_t k2;  // hi(A * C0) ^ b[1], C0 = hi(B * step) ^ a[0]  (round 1, word 2)
    uint32_t k4;  // lo(A * C0) ^ b[2]                   (round 2, word 2)
    uint32_t a[10], b[10];
};

constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;

__device__ __forceinline__ uint4 philox_blk(uint32_t blk, const PhiloxStep &k) {
    // round 0: (blk, 0, step, 0)
    uint64_t pa = static_cast<uint64_t>(kMulA) * blk;
    const uint32_t x2 = static_cast<uint32_t>(pa >> 32) ^ k.b0;
    const uint32_t x3 = static_cast<uint32_t>(pa);
    // round 1: (C0, lo(B step), x2, x3)
    uint64_t pb = static_cast<uint64_t>(kMulB) * x2;
    uint4 c = make_uint4(static_cast<uint32_t>(pb >> 32) ^ k.k1, static_cast<uint32_t>(pb),
                         x3 ^ k.k2, 0u);
    // round 2: word 3 of the input is the constant lo(A * C0)
    pa = static_cast<uint64_t>(kMulA) * c.x;
    pb = static_cast<uint64_t>(kMulB) * c.z;
    c = make_uint4(static_cast<uint32_t>(pb >> 32) ^ c.y ^ k.a[2], static_cast<uint32_t>(pb),
                   static_cast<uint32_t>(pa >> 32) ^ k.k4, static_cast<uint32_t>(pa));
#pragma unroll
    for (int r = 3; r < 10; ++r) {
        pa = static_cast<uint64_t>(kMulA) * c.x;
        pb = static_cast<uint64_t>(kMulB) * c.z;
        c = make_uint4(static_cast<uint32_t>(pb >> 32) ^ c.y ^ k.a[r], static_cast<uint32_t>(pb),
                       static_cast<uint32_t>(pa >> 32) ^ c.w ^ k.b[r], static_cast<uint32_t>(pa));
    }
    return c;
}

// min(m, |a|, |b|) in one three-input minimum.
__device__ __forceinline__ float min_abs3(float m, float a, float b) {
    float r;
    asm("{\n\t.reg .f32 x, y;\n\tabs.f32 x, %2;\n\tabs.f32 y, %3;\n\tmin.f32 %0, %1, x, y;\n\t}"
        : "=f"(r)
        : "f"(m), "f"(a), "f"(b));
    return r;
}

// max(|a|, |b|, |c|) in one three-input maximum.
__device__ __forceinline__ float max_abs3(float a, float b, float c) {
    float r;
    asm("{\n\t.reg .f32 x, y, z;\n\tabs.f32 x, %1;\n\tabs.f32 y, %2;\n\tabs.f32 z, %3;\n\t"
        "max.f32 %0, x, y, z;\n\t}"
        : "=f"(r)
        : "f"(a), "f"(b), "f"(c));
    return r;
}

// 1 / d within one ulp for d in [2^-125, 2^125]: the hardware approximation and
// one Newton-Raphson step (the decisions below allow for one ulp).
__device__ __forceinline__ float recip(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    const float e = __fmaf_rn(-d, r, 1.0f);
    return __fmaf_rn(r, e, r);
}

// --------------------------------------------------------------- ternary

// Codes of the 8 elements of a lane slot (element c in bits 2c, 2c+1).
//   pa1 = fl(|v| * rinv + 1)              one fma
//   f   = 1 + (w >> 9) * 2^-23            the draw's top 23 bits as a mantissa
//   d   = f - pa1                         exact (both in [1, 2])
// d differs from u - fl(|v| / s) by less than 2^-21 (rinv's ulp and the fma's
// rounding, 2^-22 together; the draw's dropped 24th bit; the quotient's own
// rounding), so
// keep = [d < 0] is the exact decision whenever |d| > 2^-20; otherwise `near`
// is set and the slot is recomputed with the division.
// Code bits, keep decided: b0 = !keep, b1 = keep & [v > 0] (a kept v is not
// zero).  With E = fl(d + 2): bit 30 of E is [E >= 2] = !keep (|d| > 2^-20) and
// its bit 31 is 0; bit 31 of d is keep and its bit 30 is 0 (|d| < 2).  So bits
// 31..30 of E | (d & ~v) are (b1, b0), and one funnel shift moves them in.
__device__ __forceinline__ uint32_t ternary_field8(const uint4 &raw, const uint4 &r0,
                                                   const uint4 &r1, float rinv, bool &near) {
    constexpr float kNear = 0x1p-20f;
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    const uint32_t h[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t field = 0u;
    float m = 1.0f;  // min |d| over the slot (|d| < 1)
#pragma unroll
    for (int c = 7; c >= 0; c -= 2) {
        float d2[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int cc = c - t;
            const float v = (cc & 1) ? bf16_sub<1>(h[cc >> 1], 0.0f) : bf16_sub<0>(h[cc >> 1], 0.0f);
            const float pa1 = __fmaf_rn(fabsf(v), rinv, 1.0f);
            const float f = __uint_as_float(__funnelshift_r(w[cc], 0x7Fu, 9));  // 0x3F800000 | w >> 9
            const float d = __fsub_rn(f, pa1);
            const float e = __fadd_rn(d, 2.0f);
            const uint32_t y = __float_as_uint(e) | (__float_as_uint(d) & ~__float_as_uint(v));
            field = __funnelshift_l(y, field, 2);
            d2[t] = d;
        }
        m = min_abs3(m, d2[0], d2[1]);
    }
    near = m <= kNear;
    return field;
}

// ------------------------------------------------------------------- 8 bit

__device__ __forceinline__ float bf16_at(uint32_t w, int c) {
    return __uint_as_float(c ? (w & 0xFFFF0000u) : (w << 16));
}

// Codes of the 8 elements of a lane slot, four per word.  With d = fl(v - mn),
// the exact product d * rinv is within 2^-22 t (t <= 255 (1 + 2^-22)) of the
// IEEE quotient t = fl(d / scale) (rinv's ulp and t's own rounding), so its
// nearest integer is rint(t) unless it lies within 2^-13 of a half-integer.
// y = fl(d * rinv + 1.5 * 2^23), one fma, is that nearest integer (ties to
// even) in its low mantissa bits, so the low byte of y's pattern is the code:
// three byte permutes pack four.  The distance to it, fl(d * rinv - (y - 1.5 *
// 2^23)), is one more fma; `near` is set when some distance reaches
// 1/2 - 2^-12.
__device__ __forceinline__ void u8_fields(const uint4 &raw, float mn, float rinv, uint32_t &f0,
                                          uint32_t &f1, bool &near) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const uint32_t h[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t y[8];
    float dist[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float d = (c & 1) ? bf16_sub<1>(h[c >> 1], mn) : bf16_sub<0>(h[c >> 1], mn);
        const float yf = __fmaf_rn(d, rinv, kMagic);
        y[c] = __float_as_uint(yf);
        dist[c] = __fmaf_rn(d, rinv, -__fsub_rn(yf, kMagic));
    }
    float worst = max_abs3(max_abs3(dist[0], dist[1], dist[2]), dist[3], dist[4]);
    worst = max_abs3(worst, dist[5], dist[6]);
    worst = fmaxf(worst, fabsf(dist[7]));
    f0 = __byte_perm(__byte_perm(y[0], y[1], 0x0040), __byte_perm(y[2], y[3], 0x0040), 0x5410);
    f1 = __byte_perm(__byte_perm(y[4], y[5], 0x0040), __byte_perm(y[6], y[7], 0x0040), 0x5410);
    near = worst >= 0.5f - 0x1p-12f;
}

// The ternary codes of a lane slot with the IEEE division (the slot that the
// division-free decision could not settle); out of line, so that its registers
// do not count against the common path's.
__device__ __noinline__ uint32_t ternary_slot_exact(uint4 raw, float s, uint64_t i0,
                                                    const EncodeParams &P) {
    float u[8];
    uniform4(i0, P.step, P.keys, u);
    uniform4(i0 + 4, P.step, P.keys, u + 4);
    const BucketParams bp{s, 0.0f};
    const uint32_t h[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t field = 0u;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        field |= code_exact<kTernary, 2, true>(bf16_at(h[c >> 1], c & 1), u[c], bp) << (2 * c);
    return field;
}

// ------------------------------------------------------------------ kernel

// The segment that owns launch tile `tile` (the segments' first tiles ascend).
__device__ __forceinline__ uint32_t segment_of(const EncodeSegs &S, uint64_t tile) {
    uint32_t lo = 0, hi = S.nseg;
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        if (S.s[mid].tile0 <= tile) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void issue_tile(const EncodeSegs &S, uint64_t tile, unsigned char *stage,
                                           uint64_t *bar) {
    const EncodeSeg &sg = S.s[segment_of(S, tile)];
    const uint64_t t0 = (tile - sg.tile0) * kTile;
    const uint64_t tcnt = min(static_cast<uint64_t>(kTile), sg.n - t0);
    const uint32_t gb = floor16(tcnt * 2u);
    mbar_arrive_expect_tx(bar, gb);
    if (gb) bulk_load(stage, static_cast<const uint16_t *>(sg.grad) + t0, gb, bar);
}

// A bucket that is not whole and staged (the array's last one): element-wise
// from global memory with the exact division; every lane writes whole code words.
template <int KIND>
__device__ __noinline__ void encode_partial_bucket(const EncodeParams &P, const EncodeSeg &sg,
                                                   uint64_t k, uint64_t b0, uint32_t cnt, int lane) {
    const uint16_t *g = static_cast<const uint16_t *>(sg.grad);
    constexpr int SCHEME = KIND == kU8 ? kUniform : kTernary;
    constexpr int BITS = KIND == kU8 ? 8 : 2;
    constexpr bool SR = KIND == kTern;
    Stats<SCHEME> st;
    st.init();
    for (uint32_t j = lane; j < cnt; j += 32) st.add(bf16_bits_to_float(g[b0 + j]));
    st.warp_reduce();
    const BucketParams bp = Finish<SCHEME, BITS>::run(st, cnt);
    constexpr uint32_t per = 32 / BITS;
    const uint32_t words = (cnt + per - 1) / per;
    for (uint32_t wi = lane; wi < words; wi += 32) {
        uint32_t word = 0u;
        for (uint32_t c = 0; c < per; ++c) {
            const uint32_t j = wi * per + c;
            if (j < cnt) {
                const float u = SR ? uniform1(sg.index_base + b0 + j, P.step, P.keys) : 0.0f;
                word |= code_exact<SCHEME, BITS, SR>(bf16_bits_to_float(g[b0 + j]), u, bp) << (c * BITS);
            }
        }
        sg.codes[b0 / per + wi] = word;
    }
    if (lane == 0) store_meta<SCHEME>(sg.scale, sg.offset, k, bp);
}

template <int KIND>
__global__ void __launch_bounds__(kBlock, 3) encode_bf16_fast_kernel(const __grid_constant__ EncodeParams P,
                                                                   const __grid_constant__ PhiloxStep K,
                                                                   const __grid_constant__ EncodeSegs S,
                                                                   const uint64_t ntiles) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint32_t *done = reinterpret_cast<uint32_t *>(full + kStages);  // warps done with a stage
    uint32_t *issued = done + kStages;                               // tiles issued into a stage

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the folded Philox keys in registers for the whole kernel (the smem limit
    // leaves three blocks per SM, so registers are not what bounds occupancy)
    PhiloxStep Kr;
    if constexpr (KIND == kTern) Kr = K;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0u;
            issued[s] = 0u;
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < kStages; ++s) {
            const uint64_t tile = blockIdx.x + static_cast<uint64_t>(s) * gridDim.x;
            if (tile < ntiles) {
                issue_tile(S, tile, smem + s * kStageBytes, &full[s]);
                issued[s] = 1u;
            }
        }
    }

    uint32_t it = 0;
    bool failed = false;
    for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
        const uint32_t s = it % kStages;
        const uint32_t parity = (it / kStages) & 1u;
        const unsigned char *stage = smem + s * kStageBytes;
        // the warp agrees on the wait's outcome, so its shuffles stay whole
        if (!__all_sync(kFull, mbar_wait(&full[s], parity))) {
            failed = true;
            break;
        }
        const EncodeSeg &sg = S.s[segment_of(S, tile)];
        const uint64_t lt = tile - sg.tile0;  // the tile within its segment
        const uint64_t t0 = lt * kTile;
        const uint32_t tcnt = static_cast<uint32_t>(min(static_cast<uint64_t>(kTile), sg.n - t0));
        const uint32_t staged = floor16(static_cast<uint64_t>(tcnt) * 2u) / 2u;
        // the warp's buckets of the tile, kWarps apart, so that the tile's
        // bookkeeping (wait, segment, counts, refill) is paid once for several
        for (uint32_t bb = 0; bb < kPerWarp; ++bb) {
            const uint32_t b_off = (bb * kWarps + static_cast<uint32_t>(warp)) * kB;
            const uint32_t cnt = b_off < tcnt ? min(kB, tcnt - b_off) : 0u;
            const uint64_t b0 = t0 + b_off;            // the bucket's first element in its segment
            const uint64_t d0 = sg.index_base + b0;    // ... and its draw index
            const uint64_t k = lt * (kWarps * kPerWarp) + bb * kWarps + warp;

            if (cnt == kB && b_off + kB <= staged) {
                auto slot = [&](int sl) {
                    return *reinterpret_cast<const uint4 *>(stage + (b_off + (sl * 32 + lane) * 8u) * 2u);
                };
                if constexpr (KIND == kTern) {
                    // ---- s = max |x|, on packed pairs (only the magnitudes count)
                    uint32_t a = 0u;
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {
                        const uint4 r = slot(sl);
                        a = absmax_bf16x2(a, absmax_bf16x2(r.x, r.y));
                        a = absmax_bf16x2(a, absmax_bf16x2(r.z, r.w));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) a = absmax_bf16x2(a, __shfl_xor_sync(kFull, a, o));
                    a &= 0x7FFF7FFFu;
                    const float s_ = fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u));
                    const bool fast = s_ >= 0x1p-125f && s_ <= 0x1p125f;
                    const float rinv = fast ? recip(s_) : 0.0f;
                    // ---- codes, 8 elements per slot, two lanes per code word; the slot
                    // is read from the stage again rather than kept in registers
                    // per-bucket bases: slot sl of the lane is element j = 256 sl + 8 lane,
                    // its Philox blocks (d0 + j) / 4 (draws < 2^34; d0 % 4 == 0), its
                    // code word (b0 + j) / 16
                    const uint32_t blk0 = static_cast<uint32_t>(d0 >> 2) + 2u * static_cast<uint32_t>(lane);
                    const unsigned char *src = stage + (b_off + 8u * static_cast<uint32_t>(lane)) * 2u;
                    uint32_t *dst = sg.codes + (b0 >> 4) + (lane >> 1);
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {
                        const uint32_t blk = blk0 + 64u * sl;
                        const uint4 da = philox_blk(blk, Kr), db = philox_blk(blk + 1u, Kr);
                        const uint4 r = lds128(src + 512u * sl);
                        uint32_t field = 0u;
                        bool near = true;
                        if (fast) field = ternary_field8(r, da, db, rinv, near);
                        if (near) field = ternary_slot_exact(r, s_, d0 + 256u * sl + 8u * lane, P);  // rare
                        field |= __shfl_down_sync(kFull, field, 1) << 16;
                        if ((lane & 1) == 0) __stcs(dst + 16 * sl, field);
                    }
                    if (lane == 0) sg.scale[k] = s_;
                } else {
                    uint4 raw[4];
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) raw[sl] = slot(sl);
                    // ---- min and max, on packed pairs
                    uint32_t lo = min_bf16x2(raw[0].x, raw[0].y), hi = max_bf16x2(raw[0].x, raw[0].y);
                    lo = min_bf16x2(lo, min_bf16x2(raw[0].z, raw[0].w));
                    hi = max_bf16x2(hi, max_bf16x2(raw[0].z, raw[0].w));
#pragma unroll
                    for (int sl = 1; sl < 4; ++sl) {
                        lo = min_bf16x2(lo, min_bf16x2(raw[sl].x, raw[sl].y));
                        hi = max_bf16x2(hi, max_bf16x2(raw[sl].x, raw[sl].y));
                        lo = min_bf16x2(lo, min_bf16x2(raw[sl].z, raw[sl].w));
                        hi = max_bf16x2(hi, max_bf16x2(raw[sl].z, raw[sl].w));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        lo = min_bf16x2(lo, __shfl_xor_sync(kFull, lo, o));
                        hi = max_bf16x2(hi, __shfl_xor_sync(kFull, hi, o));
                    }
                    Stats<kUniform> st;
                    st.mn = fminf(__uint_as_float(lo << 16), __uint_as_float(lo & 0xFFFF0000u));
                    st.mx = fmaxf(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
                    const BucketParams bp = Finish<kUniform, 8>::run(st, kB);
                    const bool fast = bp.scale >= 0x1p-125f && bp.scale <= 0x1p125f;
                    const float rinv = fast ? recip(bp.scale) : 0.0f;
                    uint2 *dst = reinterpret_cast<uint2 *>(sg.codes + (b0 >> 2)) + lane;  // slot sl: + 32 sl
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {
                        uint32_t f0 = 0u, f1 = 0u;
                        bool near = true;
                        if (fast) u8_fields(raw[sl], bp.a, rinv, f0, f1, near);
                        if (near) {  // rare: the flagged elements with the division
                            const uint32_t h[4] = {raw[sl].x, raw[sl].y, raw[sl].z, raw[sl].w};
                            uint32_t redo = 0xFFu;  // scales outside the fast range: all eight
                            if (fast) {
                                // with bf16 data a flagged slot holds one or two elements
                                // near a half-integer (often an exact tie of the quotient)
                                constexpr float kMagic = 12582912.0f;
                                redo = 0u;
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    const float d = (c & 1) ? bf16_sub<1>(h[c >> 1], bp.a) : bf16_sub<0>(h[c >> 1], bp.a);
                                    const float yf = __fmaf_rn(d, rinv, kMagic);
                                    const float dist = __fmaf_rn(d, rinv, -__fsub_rn(yf, kMagic));
                                    redo |= (fabsf(dist) >= 0.5f - 0x1p-12f ? 1u : 0u) << c;
                                }
                            }
                            while (redo != 0u) {  // a loop, so the common path is not predicated with it
                                const int c = __ffs(redo) - 1;
                                redo &= redo - 1u;
                                const uint32_t hw = c < 2 ? h[0] : c < 4 ? h[1] : c < 6 ? h[2] : h[3];
                                const float v = __uint_as_float((c & 1) ? (hw & 0xFFFF0000u) : (hw << 16));
                                const uint32_t code = code_exact<kUniform, 8, false>(v, 0.0f, bp);
                                const uint32_t sh = 8u * static_cast<uint32_t>(c & 3);
                                if (c < 4) f0 = (f0 & ~(0xFFu << sh)) | (code << sh);
                                else f1 = (f1 & ~(0xFFu << sh)) | (code << sh);
                            }
                        }
                        __stcs(dst + 32 * sl, make_uint2(f0, f1));
                    }
                    if (lane == 0) {
                        sg.scale[k] = bp.scale;
                        sg.offset[k] = bp.a;
                    }
                }
            } else if (cnt) {
                encode_partial_bucket<KIND>(P, sg, k, b0, cnt, lane);
            }
        }
        // this warp is done with the stage (its reads have returned: their values
        // are used above); the warp that completes the count refills the stage
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const uint32_t before = atomicAdd(&done[s], 1u);
            if (before % kWarps == kWarps - 1) {
                __threadfence_block();
                fence_proxy_async_shared();  // generic reads before the bulk copy's writes
                const uint64_t next = tile + static_cast<uint64_t>(kStages) * gridDim.x;
                if (next < ntiles) {
                    issue_tile(S, next, smem + s * kStageBytes, &full[s]);
                    issued[s] += 1u;
                }
            }
        }
    }
    if (failed && lane == 0) report_failure(&g_encode_bf16_fast_errors, P.status, kErrPipelineTimeout);
    // A warp that gave up leaves its stages unrefilled, so the other warps' waits
    // run out too; every warp gets here.  Copies still in flight (only after a
    // failure) must land before the block's shared memory goes away.
    __syncthreads();
    if (threadIdx.x == 0) {
        for (uint32_t d = 0; d < kStages; ++d)
            if (issued[d]) mbar_wait(&full[d], (issued[d] - 1u) & 1u);
    }
}

PhiloxStep philox_step(const EncodeParams &p) {
    PhiloxStep k;
    for (int r = 0; r < 10; ++r) {
        k.a[r] = p.keys.a[r];
        k.b[r] = p.keys.b[r];
    }
    const uint64_t pb0 = static_cast<uint64_t>(kMulB) * p.step;
    const uint32_t c0 = static_cast<uint32_t>(pb0 >> 32) ^ k.a[0];
    const uint64_t pa1 = static_cast<uint64_t>(kMulA) * c0;
    k.b0 = k.b[0];
    k.k1 = static_cast<uint32_t>(pb0) ^ k.a[1];
    k.k2 = static_cast<uint32_t>(pa1 >> 32) ^ k.b[1];
    k.k4 = static_cast<uint32_t>(pa1) ^ k.b[2];
    return k;
}

template <int KIND>
cudaError_t launch_one(const EncodeParams &p, const EncodeSegs &S, uint64_t ntiles,
                       cudaStream_t stream) {
    auto fn = &encode_bf16_fast_kernel<KIND>;
    const size_t smem = kSmem;
    cudaError_t e = prepare_dynamic_smem(reinterpret_cast<const void *>(fn), smem);
    if (e != cudaSuccess) return e;
    const int grid = persistent_grid(reinterpret_cast<const void *>(fn), kBlock, ntiles, smem);
    fn<<<grid, kBlock, smem, stream>>>(p, philox_step(p), S, ntiles);
    return cudaGetLastError();
}

}  // namespace

uint64_t encode_bf16_fast_tiles(uint64_t n) { return (n + kTile - 1) / kTile; }

bool encode_bf16_fast_applies(const EncodeParams &p, int scheme, int bits, int stochastic,
                              bool grad16, bool codes8) {
    // draws are indexed in 32-bit Philox blocks of four: index_base + n < 2^34
    if (!grad16 || p.err != nullptr || p.bucket != kB ||
        p.index_base + p.n >= (static_cast<uint64_t>(1) << 34))
        return false;
    if (scheme == kTernary) return stochastic != 0;
    return scheme == kUniform && bits == 8 && !stochastic && codes8;
}

cudaError_t launch_encode_bf16_fast(const EncodeParams &p, int scheme, cudaStream_t stream,
                                    const EncodeSegs *segs) {
    const EncodeSegs S = segs ? *segs : single_segment(p);
    uint64_t ntiles = 0;
    for (uint32_t i = 0; i < S.nseg; ++i) ntiles = S.s[i].tile0 + encode_bf16_fast_tiles(S.s[i].n);
    return scheme == kTernary ? launch_one<kTern>(p, S, ntiles, stream)
                              : launch_one<kU8>(p, S, ntiles, stream);
}

QC_DEFINE_TAKE_FLAG(take_encode_bf16_fast_errors, g_encode_bf16_fast_errors)

}  // namespace qc
