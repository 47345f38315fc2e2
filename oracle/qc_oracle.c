/*
 * qc_oracle.c -- plain, slow, scalar CPU oracle for the communication codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant generator with the CUDA
 * library; the two are independent restatements of the same method.
 *
 * Sources (web pages on quantized communication for distributed training):
 *   [p1] "Quantized Communication for Distributed Training" (edmondo-vault),
 *        sections "Where Quantization Sits" and "Numeric Example":
 *        quantize for the wire, dequantize on the receiver, FP32 -> FP8 payloads
 *        of embedding lookups (1,000,000 x 128 values).
 *   [p2] "Gradient quantization for communication" (chipfoundryservices),
 *        sections "How Gradient Quantization Works" and "Quantization Schemes".
 *   [p3] "Quantization for Communication" (chipfoundryservices), sections
 *        "Quantization Schemes" (uniform min/max formulas, stochastic rounding),
 *        "Quantized SGD Algorithms" (TernGrad, SignSGD majority vote),
 *        "Error Feedback for Quantization", "Quantization-Aware All-Reduce"
 *        (accumulate in higher precision), "Hardware Acceleration" (packed words).
 *   [p4] "Gradient Compression and Quantised Collectives" (praveentn.live),
 *        sections "Why sparsification fights the all-reduce" (signSGD majority
 *        vote) and "Error feedback is the component that makes it work".
 *
 * Arithmetic: IEEE-754 binary32, round-to-nearest-even, one rounding per
 * operation as written (build with -ffp-contract=off, never -ffast-math); fp64
 * only for the sign scheme's mean and exact integer arithmetic for the QSGD norm,
 * as stated there.  Each function takes the
 * steps of the method in the order the pages give them, element by element in
 * index order.  Readings taken where the pages are silent are stated at each
 * step.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

enum { ORC_SCHEME_UNIFORM = 0, ORC_SCHEME_SIGN = 1, ORC_SCHEME_TERNARY = 2, ORC_SCHEME_QSGD = 3,
       ORC_SCHEME_UNIFORM_CLIP = 4, ORC_SCHEME_LOG = 5 };
enum { ORC_ROUND_NEAREST = 0, ORC_ROUND_STOCHASTIC = 1 };
enum { ORC_DTYPE_F32 = 0, ORC_DTYPE_BF16 = 1 };
enum { ORC_OUT_MEAN = 1, ORC_ACCUMULATE_INTO_OUT = 2 };

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, written from Salmon, Moraes, Dror and Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3" (SC'11): a 4-word counter and a 2-word key,
 * ten rounds.  Each round multiplies counter words 0 and 2 by the two round
 * constants, and builds the new counter from the high halves xor-ed with the
 * other two counter words and the key, and from the low halves.  Between
 * rounds the key is bumped by the two Weyl constants (golden ratio and
 * sqrt(3)-1 in 32-bit fixed point). */

static void orc_mul_hi_lo(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo)
{
    uint64_t product = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(product >> 32);
    *lo = (uint32_t)product;
}

ORC_API void oracle_philox4x32_10(const uint32_t counter[4], const uint32_t key[2],
                                  uint32_t out[4])
{
    uint32_t x0 = counter[0], x1 = counter[1], x2 = counter[2], x3 = counter[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u; /* Weyl increment, key word 0 */
            k1 += 0xBB67AE85u; /* Weyl increment, key word 1 */
        }
        uint32_t hi0, lo0, hi2, lo2;
        orc_mul_hi_lo(0xD2511F53u, x0, &hi0, &lo0);
        orc_mul_hi_lo(0xCD9E8D57u, x2, &hi2, &lo2);
        uint32_t y0 = hi2 ^ x1 ^ k0;
        uint32_t y1 = lo2;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0;
        x1 = y1;
        x2 = y2;
        x3 = y3;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

/* The uniform draw u_i in [0, 1) used for stochastic rounding of element i.
 * The pages only say "probabilistic rounding"; the reading taken here is:
 *   key     = (low 32 bits of seed, high 32 bits of seed)
 *   counter = (low 32 of i/4, high 32 of i/4, step, 0)
 *   u_i     = (word (i mod 4) of the Philox output >> 8) * 2^-24   (exact)
 * so one Philox call serves four consecutive elements and the draw depends only
 * on (seed, step, global element index). */
ORC_API float oracle_uniform(uint64_t seed, uint32_t step, uint64_t index)
{
    uint64_t block = index >> 2;
    uint32_t counter[4] = {(uint32_t)block, (uint32_t)(block >> 32), step, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(counter, key, r);
    return (float)(r[index & 3u] >> 8) * 0x1p-24f;
}

/* ------------------------------------------------------------------------ */
/* Helpers with no codec arithmetic in them. */

static float orc_load_grad(const void *grad, int dtype, size_t i)
{
    if (dtype == ORC_DTYPE_F32)
        return ((const float *)grad)[i];
    /* bf16 -> fp32 is an exact widening: the 16 bits are the top half. */
    uint32_t bits = (uint32_t)((const uint16_t *)grad)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* After a min/max reduction a zero result is taken as +0 (the pages are
 * silent on signed zero; this makes the reduction's result unique). */
static float orc_positive_zero(float r)
{
    return (r == 0.0f) ? 0.0f : r;
}

static int orc_valid_bucket(size_t bucket)
{
    return bucket >= 32 && bucket % 32 == 0;
}

/* Packing (p3 "Hardware Acceleration", packed formats): code i of a b-bit
 * stream goes to word i / (32/b) at bit offset (i mod (32/b)) * b, least
 * significant bits first (bit order within a word: a reading). */
static void orc_put_code(uint32_t *words, size_t i, int bits, uint32_t code)
{
    size_t per_word = (size_t)(32 / bits);
    words[i / per_word] |= code << ((i % per_word) * (size_t)bits);
}

static uint32_t orc_get_code(const uint32_t *words, size_t i, int bits)
{
    size_t per_word = (size_t)(32 / bits);
    uint32_t mask = (bits == 32) ? 0xFFFFFFFFu : ((1u << bits) - 1u);
    return (words[i / per_word] >> ((i % per_word) * (size_t)bits)) & mask;
}

ORC_API size_t oracle_code_words(size_t n, int bits)
{
    return (n * (size_t)bits + 31) / 32;
}

ORC_API size_t oracle_num_buckets(size_t n, size_t bucket)
{
    return (n + bucket - 1) / bucket;
}

/* ------------------------------------------------------------------------ */
/* Uniform min/max quantization with optional error feedback.
 *
 * p3 "Quantization Schemes": scale = (max - min) / (2^bits - 1),
 * q = round((x - min) / scale), x ~= q * scale + min; stochastic rounding takes
 * floor((x - min)/scale) with probability 1 - frac and the ceiling with
 * probability frac.  p3 "Error Feedback for Quantization" and p4 "Error
 * feedback ...": e = e + grad; q = quantize(e); e = e - dequantize(q).
 *
 * Per bucket k of `bucket` elements (the last may be partial):
 *   p_i   = e_i + g_i                 (or g_i without error feedback)
 *   mn, mx = min p, max p             (zero taken as +0)
 *   scale = (mx - mn) / L,  L = 2^bits - 1          (IEEE division)
 *   scale == 0  -> q_i = 0            (constant bucket: a reading)
 *   t_i   = (p_i - mn) / scale
 *   nearest:    q_i = min(rint(t_i), L)             (ties to even: a reading)
 *   stochastic: q_i = min(floor(t_i) + [u_i < t_i - floor(t_i)], L)
 *   deq_i = fma(q_i, scale, mn)       (one rounding: a reading)
 *   e_i   = p_i - deq_i
 * Outputs: packed codes, scale[k], offset[k] = mn.
 *
 * `index_base` is the global index of element 0 of this slice (it must start
 * on a bucket boundary); the stochastic draw uses global indices, so a slice
 * reproduces exactly the corresponding part of a whole-array call. */
ORC_API int oracle_encode_uniform(const void *grad, int dtype, float *err, size_t n,
                                  uint64_t index_base, int bits, size_t bucket, int mode,
                                  uint64_t seed, uint32_t step, uint32_t *codes,
                                  float *scale_out, float *offset_out)
{
    if (!(bits == 1 || bits == 2 || bits == 4 || bits == 8) || !orc_valid_bucket(bucket))
        return -1;
    const uint32_t L = (1u << bits) - 1u;
    const float Lf = (float)L;
    memset(codes, 0, oracle_code_words(n, bits) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    if (!p)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
        }
        float mn = p[0], mx = p[0];
        for (size_t j = 1; j < cnt; ++j) {
            if (p[j] < mn)
                mn = p[j];
            if (p[j] > mx)
                mx = p[j];
        }
        mn = orc_positive_zero(mn);
        mx = orc_positive_zero(mx);
        float range = mx - mn;
        float scale = range / Lf;
        for (size_t j = 0; j < cnt; ++j) {
            uint32_t q = 0;
            if (scale != 0.0f) {
                float diff = p[j] - mn;
                float t = diff / scale;
                float level;
                if (mode == ORC_ROUND_NEAREST) {
                    level = rintf(t);
                } else {
                    float f = floorf(t);
                    float frac = t - f;
                    float u = oracle_uniform(seed, step, index_base + lo + j);
                    level = (u < frac) ? f + 1.0f : f;
                }
                if (!(level >= 0.0f)) /* non-finite input: unspecified, never UB */
                    level = 0.0f;
                q = (level > Lf) ? L : (uint32_t)level;
            }
            orc_put_code(codes, lo + j, bits, q);
            if (err) {
                float deq = fmaf((float)q, scale, mn);
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = scale;
        offset_out[k] = mn;
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Uniform quantization over a percentile-clipped range, with error feedback.
 *
 * p3 "Adaptive Quantization Strategies", Percentile Clipping: outliers are
 * clipped before quantizing by setting min and max to the 1st and 99th
 * percentiles instead of the absolute extremes.  Readings: the percentile is
 * the nearest-rank one (the value of rank ceil(P * cnt / 100) in the sorted
 * bucket, 1-based), so both bounds are elements of the bucket:
 *   k_lo = ceil(cnt / 100) - 1,  k_hi = ceil(99 * cnt / 100) - 1   (0-based)
 *   mn = sorted(p)[k_lo],  mx = sorted(p)[k_hi]     (zero taken as +0)
 * Every element is clamped into [mn, mx] and then quantized exactly as in
 * oracle_encode_uniform with these mn and mx; the dequantized value is that of
 * the clamped element, so the error-feedback residual e = p - deq carries the
 * clipped part.  Buckets of at most 99 elements have k_lo = 0, k_hi = cnt - 1:
 * the absolute min and max.  Decoding is the uniform decode. */
static int orc_cmp_float(const void *a, const void *b)
{
    float x = *(const float *)a, y = *(const float *)b;
    return (x > y) - (x < y);
}

ORC_API int oracle_encode_uniform_clip(const void *grad, int dtype, float *err, size_t n,
                                       uint64_t index_base, int bits, size_t bucket, int mode,
                                       uint64_t seed, uint32_t step, uint32_t *codes,
                                       float *scale_out, float *offset_out)
{
    if (!(bits == 1 || bits == 2 || bits == 4 || bits == 8) || !orc_valid_bucket(bucket))
        return -1;
    const uint32_t L = (1u << bits) - 1u;
    const float Lf = (float)L;
    memset(codes, 0, oracle_code_words(n, bits) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    float *sorted = (float *)malloc(bucket * sizeof(float));
    if (!p || !sorted) {
        free(p);
        free(sorted);
        return -2;
    }
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
            sorted[j] = p[j];
        }
        qsort(sorted, cnt, sizeof(float), orc_cmp_float);
        size_t k_lo = (cnt + 99) / 100 - 1;
        size_t k_hi = (99 * cnt + 99) / 100 - 1;
        float mn = orc_positive_zero(sorted[k_lo]);
        float mx = orc_positive_zero(sorted[k_hi]);
        float range = mx - mn;
        float scale = range / Lf;
        for (size_t j = 0; j < cnt; ++j) {
            float pc = p[j] < mn ? mn : (p[j] > mx ? mx : p[j]);
            uint32_t q = 0;
            if (scale != 0.0f) {
                float diff = pc - mn;
                float t = diff / scale;
                float level;
                if (mode == ORC_ROUND_NEAREST) {
                    level = rintf(t);
                } else {
                    float f = floorf(t);
                    float frac = t - f;
                    float u = oracle_uniform(seed, step, index_base + lo + j);
                    level = (u < frac) ? f + 1.0f : f;
                }
                if (!(level >= 0.0f))
                    level = 0.0f;
                q = (level > Lf) ? L : (uint32_t)level;
            }
            orc_put_code(codes, lo + j, bits, q);
            if (err) {
                float deq = fmaf((float)q, scale, mn);
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = scale;
        offset_out[k] = mn;
    }
    free(p);
    free(sorted);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Scaled sign (1-bit) with error feedback.
 *
 * p3 "Quantized SGD Algorithms" (SignSGD: the sign only) and "Bit-Width
 * Selection" (1-bit with error feedback); p4 (signSGD, error feedback).
 * The per-bucket magnitude s is the mean of |p| (a reading: the scaled-sign
 * form whose dequantized bucket keeps the l1 mass):
 *   p_i  = e_i + g_i
 *   s    = (sum over the bucket of |p_i|, in fp64, index order) / cnt,
 *          rounded once to fp32
 *   bit_i = [p_i >= 0]                 (sign(0) = +1: a reading)
 *   deq_i = bit_i ? s : -s ;  e_i = p_i - deq_i
 * Outputs: 32 sign bits per word, scale[k] = s. */
ORC_API int oracle_encode_sign(const void *grad, int dtype, float *err, size_t n, size_t bucket,
                               uint32_t *codes, float *scale_out)
{
    if (!orc_valid_bucket(bucket))
        return -1;
    memset(codes, 0, oracle_code_words(n, 1) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    if (!p)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
        }
        double sum = 0.0;
        for (size_t j = 0; j < cnt; ++j)
            sum += fabs((double)p[j]);
        float s = (float)(sum / (double)cnt);
        for (size_t j = 0; j < cnt; ++j) {
            uint32_t bit = (p[j] >= 0.0f) ? 1u : 0u;
            orc_put_code(codes, lo + j, 1, bit);
            if (err) {
                float deq = bit ? s : -s;
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = s;
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* TernGrad ternary {-1, 0, +1} with a per-bucket scale.
 *
 * p3 "Quantized SGD Algorithms": TernGrad quantizes to {-1, 0, +1} with a scale
 * factor.  The stochastic rule is the named method's (keep the sign with
 * probability |p|/s, s = max |p|); the deterministic variant keeps it when
 * |p|/s > 1/2.  Codes {-1, 0, +1} -> {0, 1, 2} in 2 bits (a reading).
 *   s = max |p| (+0 for an all-zero bucket; then every code is 1)
 *   pr_i = |p_i| / s ;  keep_i = stochastic ? [u_i < pr_i] : [pr_i > 1/2]
 *   code_i = keep_i ? (p_i > 0 ? 2 : 0) : 1 ;  deq_i = (code_i - 1) * s
 *   e_i = p_i - deq_i (with error feedback)
 * Outputs: 16 codes per word, scale[k] = s. */
ORC_API int oracle_encode_ternary(const void *grad, int dtype, float *err, size_t n,
                                  uint64_t index_base, size_t bucket, int mode, uint64_t seed,
                                  uint32_t step, uint32_t *codes, float *scale_out)
{
    if (!orc_valid_bucket(bucket))
        return -1;
    memset(codes, 0, oracle_code_words(n, 2) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    if (!p)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
        }
        float s = 0.0f;
        for (size_t j = 0; j < cnt; ++j) {
            float a = fabsf(p[j]);
            if (a > s)
                s = a;
        }
        s = orc_positive_zero(s);
        for (size_t j = 0; j < cnt; ++j) {
            uint32_t code = 1;
            if (s != 0.0f) {
                float pr = fabsf(p[j]) / s;
                int keep;
                if (mode == ORC_ROUND_NEAREST)
                    keep = pr > 0.5f;
                else
                    keep = oracle_uniform(seed, step, index_base + lo + j) < pr;
                if (keep)
                    code = (p[j] > 0.0f) ? 2u : 0u;
            }
            orc_put_code(codes, lo + j, 2, code);
            if (err) {
                float deq = (float)((int)code - 1) * s;
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = s;
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The L2 norm of a bucket, exactly rounded.
 *
 * The pages and the named method (Alistarh et al.) define QSGD's scale as the
 * norm ||v||_2 and leave its arithmetic open.  Reading: nrm is the binary32
 * value nearest (ties to even) to the square root of the EXACT sum of the
 * squares, so it depends neither on the order of the sum nor on a working
 * precision.
 *
 * Every binary32 x is m * 2^e with an integer m < 2^24 and e >= -149, so its
 * square m^2 * 2^(2e) is an integer multiple of 2^-298.  The sum is therefore
 * held exactly as an unsigned integer A in units of 2^-298, in 32-bit limbs
 * (least significant first).  The largest finite square is below 2^256, so a
 * bucket of up to 2^24 elements keeps A below 2^578. */
#define ORC_WIDE_LIMBS 24 /* 768 bits: room for A * 2^60 below */

/* w += x * 2^pos for a 32-bit x. */
static void orc_wide_add32(uint32_t *w, uint32_t x, unsigned pos)
{
    unsigned k = pos / 32;
    uint64_t t = (uint64_t)x << (pos % 32); /* spans limbs k and k + 1 */
    uint64_t s = (uint64_t)w[k] + (uint32_t)t;
    w[k] = (uint32_t)s;
    s = (uint64_t)w[k + 1] + (t >> 32) + (s >> 32);
    w[k + 1] = (uint32_t)s;
    uint64_t carry = s >> 32;
    for (unsigned j = k + 2; carry && j < ORC_WIDE_LIMBS; ++j) {
        s = (uint64_t)w[j] + carry;
        w[j] = (uint32_t)s;
        carry = s >> 32;
    }
}

/* A += x^2 / 2^-298 (exact).  Non-finite x is skipped (unspecified, never UB). */
static void orc_wide_add_square(uint32_t *A, float x)
{
    uint32_t b;
    memcpy(&b, &x, sizeof b);
    uint32_t ex = (b >> 23) & 0xFFu, m = b & 0x7FFFFFu;
    if (ex == 0xFFu)
        return;
    int e; /* |x| = m * 2^e */
    if (ex == 0) {
        e = -149;
    } else {
        m |= 0x800000u;
        e = (int)ex - 150;
    }
    uint64_t sq = (uint64_t)m * m; /* < 2^48 */
    unsigned pos = (unsigned)(2 * e + 298);
    orc_wide_add32(A, (uint32_t)sq, pos);
    orc_wide_add32(A, (uint32_t)(sq >> 32), pos + 32);
}

static int orc_wide_bit(const uint32_t *w, unsigned i)
{
    return (int)((w[i / 32] >> (i % 32)) & 1u);
}

/* a = (a << 2) | two, for a number of `nl` limbs. */
static void orc_wide_shl2_in(uint32_t *a, int nl, uint32_t two)
{
    for (int j = nl - 1; j > 0; --j)
        a[j] = (a[j] << 2) | (a[j - 1] >> 30);
    a[0] = (a[0] << 2) | two;
}

/* a = (a << 1) | one. */
static void orc_wide_shl1_in(uint32_t *a, int nl, uint32_t one)
{
    for (int j = nl - 1; j > 0; --j)
        a[j] = (a[j] << 1) | (a[j - 1] >> 31);
    a[0] = (a[0] << 1) | one;
}

static int orc_wide_geq(const uint32_t *a, const uint32_t *b, int nl)
{
    for (int j = nl - 1; j >= 0; --j)
        if (a[j] != b[j])
            return a[j] > b[j];
    return 1;
}

static void orc_wide_sub(uint32_t *a, const uint32_t *b, int nl)
{
    uint64_t borrow = 0;
    for (int j = 0; j < nl; ++j) {
        uint64_t d = (uint64_t)a[j] - b[j] - borrow;
        a[j] = (uint32_t)d;
        borrow = (d >> 63) & 1u;
    }
}

/* The binary32 value nearest (ties to even) to sqrt(A * 2^-298).
 *
 * N = A * 2^60 and R = floor(sqrt(N)) by the schoolbook digit-by-digit method
 * (two bits of N per bit of the root, remainder kept exactly), so that
 * sqrt(A * 2^-298) = (R + f) * 2^-179 with 0 <= f < 1 and f > 0 exactly when the
 * remainder is not zero.  R >= 2^30 whenever A > 0.  The result keeps the top
 * 24 bits of R (fewer below the normal range, where the quantum is 2^-149,
 * i.e. 2^30 units of R) and rounds on the next bit and the bits below it. */
static float orc_wide_sqrt_f32(const uint32_t *A)
{
    enum { NL = ORC_WIDE_LIMBS, RL = ORC_WIDE_LIMBS / 2 + 1 };
    uint32_t N[NL] = {0};
    for (int j = NL - 1; j >= 0; --j) { /* N = A << 60 */
        uint32_t v = 0;
        int src = j - 1;                 /* 60 = 32 + 28 */
        if (src >= 0)
            v |= A[src] << 28;
        if (src - 1 >= 0)
            v |= A[src - 1] >> 4;
        N[j] = v;
    }
    int top = 32 * NL - 1;
    while (top >= 0 && !orc_wide_bit(N, (unsigned)top))
        --top;
    if (top < 0)
        return 0.0f;
    uint32_t R[RL] = {0}, rem[RL] = {0}, t[RL];
    for (int i = top / 2; i >= 0; --i) {
        uint32_t two = (uint32_t)(orc_wide_bit(N, 2u * i + 1) << 1 | orc_wide_bit(N, 2u * i));
        orc_wide_shl2_in(rem, RL, two);
        memcpy(t, R, sizeof t); /* t = 4 R + 1 (R before this step) */
        orc_wide_shl2_in(t, RL, 1u);
        orc_wide_shl1_in(R, RL, 0u);
        if (orc_wide_geq(rem, t, RL)) {
            orc_wide_sub(rem, t, RL);
            R[0] |= 1u;
        }
    }
    int rbits = 32 * RL - 1;
    while (!orc_wide_bit(R, (unsigned)rbits))
        --rbits;
    rbits += 1;                                  /* bit length of R */
    int shift = rbits - 24 > 30 ? rbits - 24 : 30;
    uint32_t m = 0;
    for (int i = rbits - 1; i >= shift; --i)     /* the kept bits, at most 24 */
        m = (m << 1) | (uint32_t)orc_wide_bit(R, (unsigned)i);
    int guard = orc_wide_bit(R, (unsigned)(shift - 1));
    int sticky = 0;
    for (int i = 0; i < shift - 1; ++i)
        sticky |= orc_wide_bit(R, (unsigned)i);
    for (int j = 0; j < RL; ++j)
        sticky |= rem[j] != 0;
    if (guard && (sticky || (m & 1u)))
        m += 1; /* may carry to 2^24: still exact */
    return ldexpf((float)m, shift - 179);
}

/* QSGD: s-level stochastic quantization scaled by the bucket's L2 norm.
 *
 * p3 "Quantized SGD Algorithms" (QSGD: stochastic quantization with an unbiased
 * estimator, s levels, compression ratio 32/log2(s)); p4 "Why sparsification
 * fights the all-reduce" (QSGD preserves unbiasedness).  The level rule is the
 * named method's (Alistarh et al.): with l = floor(|v_i| / ||v|| * s), keep l
 * with probability 1 - frac and l + 1 with probability frac.  Readings: the norm
 * is taken per bucket; a b-bit code is one sign bit (top bit, set for p < 0)
 * over b-1 level bits, s = 2^(b-1) - 1; the unit ||v|| / s is rounded once and
 * the level is found like the uniform scheme's with min = 0:
 *   p_i  = e_i + g_i
 *   nrm  = sqrt(sum of p_i^2) with the sum exact and the root rounded once to
 *          binary32 (orc_wide_sqrt_f32 above)
 *   unit = nrm / s ;  unit == 0 -> every code 0
 *   t_i  = |p_i| / unit
 *   stochastic: lvl = min(floor(t_i) + [u_i < t_i - floor(t_i)], s)
 *   nearest:    lvl = min(rint(t_i), s)
 *   code = [p_i < 0] << (b-1) | lvl ;  deq_i = +-fl(lvl * unit)
 *   e_i  = p_i - deq_i
 * Outputs: packed codes, scale[k] = unit. */
ORC_API int oracle_encode_qsgd(const void *grad, int dtype, float *err, size_t n,
                               uint64_t index_base, int bits, size_t bucket, int mode,
                               uint64_t seed, uint32_t step, uint32_t *codes, float *scale_out)
{
    if (!(bits == 2 || bits == 4 || bits == 8) || !orc_valid_bucket(bucket))
        return -1;
    const uint32_t s = (1u << (bits - 1)) - 1u;
    const float sf = (float)s;
    memset(codes, 0, oracle_code_words(n, bits) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    if (!p)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
        }
        uint32_t A[ORC_WIDE_LIMBS] = {0};
        for (size_t j = 0; j < cnt; ++j)
            orc_wide_add_square(A, p[j]);
        float nrm = orc_wide_sqrt_f32(A);
        float unit = nrm / sf;
        for (size_t j = 0; j < cnt; ++j) {
            uint32_t lvl = 0;
            float a = fabsf(p[j]);
            if (unit != 0.0f) {
                float t = a / unit;
                float level;
                if (mode == ORC_ROUND_NEAREST) {
                    level = rintf(t);
                } else {
                    float f = floorf(t);
                    float frac = t - f;
                    float u = oracle_uniform(seed, step, index_base + lo + j);
                    level = (u < frac) ? f + 1.0f : f;
                }
                if (!(level >= 0.0f))
                    level = 0.0f;
                lvl = (level > sf) ? s : (uint32_t)level;
            }
            uint32_t neg = (p[j] < 0.0f) ? 1u : 0u;
            orc_put_code(codes, lo + j, bits, (neg << (bits - 1)) | lvl);
            if (err) {
                float mag = (float)lvl * unit;
                float deq = neg ? -mag : mag;
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = unit;
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Logarithmic (non-uniform) quantization with error feedback.
 *
 * p3 "Quantization Schemes" (Non-Uniform Quantization: logarithmic levels, more
 * levels near zero, dequantization through a lookup table).  Readings: a b-bit
 * code is one sign bit (top, set for p < 0) over b-1 level bits j; with
 * J = 2^(b-1) - 1 the level magnitudes are 0 (j = 0) and s * 2^(j - J)
 * (j = 1 .. J), s = max |p| over the bucket (zero taken as +0), so each level
 * below the top is half the next; x = fl(|p| / s) is placed between its two
 * adjacent levels and rounded to the nearer (ties to the even level index) or,
 * stochastically, up with probability equal to its position between them (the
 * rule the pages give for stochastic rounding, unbiased):
 *   x >= 1:               j = J
 *   2^(1-J) <= x < 1:     lower level 2^e (e = floor(log2 x)), m = (x - 2^e) / 2^e,
 *                         j = e + J + [m > 1/2, or m = 1/2 and e + J odd]   (nearest)
 *                         j = e + J + [u < m]                              (stochastic)
 *   x < 2^(1-J):          f = x / 2^(1-J);  j = [f > 1/2] or [u < f]
 *   s == 0:               j = 0
 *   deq = +-(j ? fl(s * 2^(j - J)) : 0) with the code's sign;  e = p - deq
 * Outputs: packed codes, scale[k] = s. */
ORC_API int oracle_encode_log(const void *grad, int dtype, float *err, size_t n,
                              uint64_t index_base, int bits, size_t bucket, int mode,
                              uint64_t seed, uint32_t step, uint32_t *codes, float *scale_out)
{
    if (!(bits == 2 || bits == 4 || bits == 8) || !orc_valid_bucket(bucket))
        return -1;
    const int J = (1 << (bits - 1)) - 1;
    const float lo1 = ldexpf(1.0f, 1 - J); /* the smallest non-zero level, in units of s */
    memset(codes, 0, oracle_code_words(n, bits) * sizeof(uint32_t));
    float *p = (float *)malloc(bucket * sizeof(float));
    if (!p)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        float s = 0.0f;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
            if (fabsf(p[j]) > s)
                s = fabsf(p[j]);
        }
        s = orc_positive_zero(s);
        for (size_t j = 0; j < cnt; ++j) {
            uint32_t neg = (p[j] < 0.0f) ? 1u : 0u;
            int lvl = 0;
            if (s != 0.0f) {
                float x = fabsf(p[j]) / s;
                float u = (mode == ORC_ROUND_STOCHASTIC)
                              ? oracle_uniform(seed, step, index_base + lo + j) : 0.0f;
                if (x >= 1.0f) {
                    lvl = J;
                } else if (x >= lo1) {
                    int ex;
                    (void)frexpf(x, &ex); /* x = fr * 2^ex, fr in [1/2, 1) */
                    float lower = ldexpf(1.0f, ex - 1);
                    float m = (x - lower) / lower;
                    int j0 = (ex - 1) + J;
                    int up = (mode == ORC_ROUND_NEAREST)
                                 ? (m > 0.5f || (m == 0.5f && (j0 & 1)))
                                 : (u < m);
                    lvl = j0 + up;
                } else {
                    float f = x / lo1;
                    lvl = (mode == ORC_ROUND_NEAREST) ? (f > 0.5f) : (u < f);
                }
            }
            orc_put_code(codes, lo + j, bits, (neg << (bits - 1)) | (uint32_t)lvl);
            if (err) {
                float mag = lvl ? s * ldexpf(1.0f, lvl - J) : 0.0f;
                float deq = neg ? -mag : mag;
                err[lo + j] = p[j] - deq;
            }
        }
        scale_out[k] = s;
    }
    free(p);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Receiver side: dequantize M workers' payloads and accumulate in fp32.
 *
 * p1 "Where Quantization Sits" (receive, dequantize, continue); p2 "How
 * Gradient Quantization Works" (dequantize, then average or sum); p3
 * "Quantization-Aware All-Reduce" (dequantize after the exchange; accumulate
 * in higher precision).  For every element i (bucket k = i / bucket):
 *   acc = +0
 *   for w = 0 .. M-1 in this order:
 *       d = uniform: fma(q, scale_w[k], offset_w[k])
 *           sign:    bit ? s_w[k] : -s_w[k]
 *           ternary: (code - 1) * s_w[k]
 *       acc = acc + d
 *   r = mean ? acc / M : acc ;  out_i = accumulate ? out_i + r : r
 * Worker w's codes start at codes + w*codes_stride_words and its metadata at
 * scale/offset + w*meta_stride. */
ORC_API int oracle_decode_accumulate(const uint32_t *codes, size_t codes_stride_words,
                                     const float *scale, const float *offset,
                                     size_t meta_stride, int M, size_t n, int bits,
                                     size_t bucket, int scheme, float *out, int flags)
{
    if (M < 1 || !orc_valid_bucket(bucket))
        return -1;
    if (scheme < ORC_SCHEME_UNIFORM || scheme > ORC_SCHEME_LOG)
        return -1;
    if (scheme == ORC_SCHEME_UNIFORM_CLIP) /* a uniform payload over the clipped range */
        scheme = ORC_SCHEME_UNIFORM;
    if (scheme == ORC_SCHEME_UNIFORM && !(bits == 1 || bits == 2 || bits == 4 || bits == 8))
        return -1;
    if (scheme == ORC_SCHEME_SIGN && bits != 1)
        return -1;
    if (scheme == ORC_SCHEME_TERNARY && bits != 2)
        return -1;
    if ((scheme == ORC_SCHEME_QSGD || scheme == ORC_SCHEME_LOG) && !(bits == 2 || bits == 4 || bits == 8))
        return -1;
    for (size_t i = 0; i < n; ++i) {
        size_t k = i / bucket;
        float acc = 0.0f;
        for (int w = 0; w < M; ++w) {
            const uint32_t *cw = codes + (size_t)w * codes_stride_words;
            uint32_t q = orc_get_code(cw, i, bits);
            float s = scale[(size_t)w * meta_stride + k];
            float d;
            if (scheme == ORC_SCHEME_UNIFORM)
                d = fmaf((float)q, s, offset[(size_t)w * meta_stride + k]);
            else if (scheme == ORC_SCHEME_SIGN)
                d = q ? s : -s;
            else if (scheme == ORC_SCHEME_TERNARY)
                d = (float)((int)q - 1) * s;
            else if (scheme == ORC_SCHEME_QSGD) { /* sign bit over the level */
                uint32_t lvl = q & ((1u << (bits - 1)) - 1u);
                float mag = (float)lvl * s;
                d = (q >> (bits - 1)) ? -mag : mag;
            } else { /* LOG: sign bit over the level; the level's power of two */
                int J = (1 << (bits - 1)) - 1;
                int lvl = (int)(q & ((1u << (bits - 1)) - 1u));
                float mag = lvl ? s * ldexpf(1.0f, lvl - J) : 0.0f;
                d = (q >> (bits - 1)) ? -mag : mag;
            }
            acc = acc + d;
        }
        float r = (flags & ORC_OUT_MEAN) ? acc / (float)M : acc;
        out[i] = (flags & ORC_ACCUMULATE_INTO_OUT) ? out[i] + r : r;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k sparsification with 8-bit quantization of the kept values and error
 * feedback, per bucket.
 *
 * p2 "Quantization Schemes" (Top-K Sparsification: send only the largest K% of
 * gradients, combined with quantization; Error Feedback: accumulate the errors
 * locally); p3 "Combination with Other Techniques" (quantize the sparse
 * gradients); p4 intro and "Why sparsification fights the all-reduce" (the
 * largest-magnitude coordinates travel as index-value pairs).  Readings: the
 * largest K are taken per bucket (like every other statistic here, and giving
 * a fixed payload per bucket); order by |p| descending, ties to the lower
 * index; the kept values are quantized with the uniform 8-bit formulas over
 * their own min..max; an element not kept stays whole in the residual.
 * Per bucket k (cnt elements, K = min(keep, cnt)):
 *   p_i = e_i + g_i (or g_i)
 *   kept = the first K of the bucket's elements ordered by (|p| desc, i asc)
 *   mn, mx = min, max of p over kept (zero taken as +0); scale = (mx - mn)/255
 *   q, deq: as oracle_encode_uniform (8 bits) for each kept element
 *   e_i = kept ? p_i - deq_i : p_i
 * Outputs: slot t < K of bucket k holds the t-th kept element in ascending
 * index order: idx[k*keep + t] = its global index (index_base + i),
 * codes[k*keep + t] = q; slots t >= K hold index 0xFFFFFFFF and code 0;
 * scale[k], offset[k] = mn. */
typedef struct {
    float mag;
    uint32_t j;
} orc_mag_index;

static int orc_cmp_topk(const void *a, const void *b)
{
    const orc_mag_index *x = (const orc_mag_index *)a, *y = (const orc_mag_index *)b;
    if (x->mag != y->mag)
        return x->mag > y->mag ? -1 : 1; /* larger magnitude first */
    return (x->j > y->j) - (x->j < y->j); /* then the lower index */
}

ORC_API int oracle_topk_encode(const void *grad, int dtype, float *err, size_t n,
                               uint64_t index_base, size_t bucket, size_t keep, int mode,
                               uint64_t seed, uint32_t step, uint32_t *idx_out,
                               uint8_t *codes_out, float *scale_out, float *offset_out)
{
    if (!orc_valid_bucket(bucket) || keep < 1 || keep > bucket)
        return -1;
    const float Lf = 255.0f;
    float *p = (float *)malloc(bucket * sizeof(float));
    orc_mag_index *order = (orc_mag_index *)malloc(bucket * sizeof(orc_mag_index));
    unsigned char *kept = (unsigned char *)malloc(bucket);
    if (!p || !order || !kept) {
        free(p);
        free(order);
        free(kept);
        return -2;
    }
    size_t nb = oracle_num_buckets(n, bucket);
    for (size_t k = 0; k < nb; ++k) {
        size_t lo = k * bucket;
        size_t cnt = (n - lo < bucket) ? (n - lo) : bucket;
        size_t K = keep < cnt ? keep : cnt;
        for (size_t j = 0; j < cnt; ++j) {
            float g = orc_load_grad(grad, dtype, lo + j);
            p[j] = err ? err[lo + j] + g : g;
            order[j].mag = fabsf(p[j]);
            order[j].j = (uint32_t)j;
            kept[j] = 0;
        }
        qsort(order, cnt, sizeof(orc_mag_index), orc_cmp_topk);
        for (size_t t = 0; t < K; ++t)
            kept[order[t].j] = 1;
        float mn = 0.0f, mx = 0.0f;
        int first = 1;
        for (size_t j = 0; j < cnt; ++j) {
            if (!kept[j])
                continue;
            if (first || p[j] < mn)
                mn = p[j];
            if (first || p[j] > mx)
                mx = p[j];
            first = 0;
        }
        mn = orc_positive_zero(mn);
        mx = orc_positive_zero(mx);
        float scale = (mx - mn) / Lf;
        size_t t = 0;
        for (size_t j = 0; j < cnt; ++j) {
            if (!kept[j]) {
                if (err)
                    err[lo + j] = p[j];
                continue;
            }
            uint32_t q = 0;
            if (scale != 0.0f) {
                float t_ = (p[j] - mn) / scale;
                float level;
                if (mode == ORC_ROUND_NEAREST) {
                    level = rintf(t_);
                } else {
                    float f = floorf(t_);
                    float frac = t_ - f;
                    float u = oracle_uniform(seed, step, index_base + lo + j);
                    level = (u < frac) ? f + 1.0f : f;
                }
                if (!(level >= 0.0f))
                    level = 0.0f;
                q = (level > Lf) ? 255u : (uint32_t)level;
            }
            idx_out[k * keep + t] = (uint32_t)(index_base + lo + j);
            codes_out[k * keep + t] = (uint8_t)q;
            ++t;
            if (err) {
                float deq = fmaf((float)q, scale, mn);
                err[lo + j] = p[j] - deq;
            }
        }
        for (; t < keep; ++t) {
            idx_out[k * keep + t] = 0xFFFFFFFFu;
            codes_out[k * keep + t] = 0;
        }
        scale_out[k] = scale;
        offset_out[k] = mn;
    }
    free(p);
    free(order);
    free(kept);
    return 0;
}

/* Receiver of top-k payloads: scatter and accumulate M workers' index-value
 * pairs into a dense fp32 vector in fixed worker order ("Why sparsification
 * fights the all-reduce": the exchange is an all-gather of index-value pairs).
 *   acc_i = +0 for every i
 *   for w = 0 .. M-1, for each bucket k, for each slot t:
 *       i = idx_w[k*keep + t]; skipped unless k*bucket <= i < min((k+1)*bucket, n)
 *       acc_i = acc_i + fma(code, scale_w[k], offset_w[k])
 *   r = mean ? acc / M : acc ;  out_i = accumulate ? out_i + r : r
 * Worker w's pairs start at w * pair_stride, its metadata at w * meta_stride. */
ORC_API int oracle_topk_decode(const uint32_t *idx, const uint8_t *codes, size_t pair_stride,
                               const float *scale, const float *offset, size_t meta_stride, int M,
                               size_t n, size_t bucket, size_t keep, float *out, int flags)
{
    if (M < 1 || !orc_valid_bucket(bucket) || keep < 1 || keep > bucket)
        return -1;
    float *acc = (float *)calloc(n ? n : 1, sizeof(float));
    if (!acc)
        return -2;
    size_t nb = oracle_num_buckets(n, bucket);
    for (int w = 0; w < M; ++w) {
        for (size_t k = 0; k < nb; ++k) {
            size_t lo = k * bucket;
            size_t hi = (n - lo < bucket) ? n : lo + bucket;
            float s = scale[(size_t)w * meta_stride + k];
            float o = offset[(size_t)w * meta_stride + k];
            for (size_t t = 0; t < keep; ++t) {
                size_t at = (size_t)w * pair_stride + k * keep + t;
                uint32_t i = idx[at];
                if (i < lo || i >= hi)
                    continue;
                acc[i] = acc[i] + fmaf((float)codes[at], s, o);
            }
        }
    }
    for (size_t i = 0; i < n; ++i) {
        float r = (flags & ORC_OUT_MEAN) ? acc[i] / (float)M : acc[i];
        out[i] = (flags & ORC_ACCUMULATE_INTO_OUT) ? out[i] + r : r;
    }
    free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* signSGD majority vote (p3 "Quantized SGD Algorithms"; p4 "Why sparsification
 * fights the all-reduce"): out bit i = [2 * (number of workers with bit i set)
 * >= M].  A tie (even M) gives 1, matching sign(0) = +1 (a reading).  Bits past
 * n in the last word are 0. */
ORC_API int oracle_sign_vote(const uint32_t *signs, size_t stride_words, int M, size_t n,
                             uint32_t *out)
{
    if (M < 1)
        return -1;
    memset(out, 0, oracle_code_words(n, 1) * sizeof(uint32_t));
    for (size_t i = 0; i < n; ++i) {
        long count = 0;
        for (int w = 0; w < M; ++w)
            count += (long)orc_get_code(signs + (size_t)w * stride_words, i, 1);
        if (2 * count >= (long)M)
            orc_put_code(out, i, 1, 1u);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (OCP 8-bit floating point, E4M3 variant): sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; the
 * largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0 encodes the
 * subnormals m * 2^-9. */

ORC_API float oracle_e4m3_to_f32(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    float v;
    if (e == 0xF && m == 0x7)
        v = NAN;
    else if (e == 0)
        v = ldexpf((float)m, -9);
    else
        v = ldexpf((float)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* fp32 -> E4M3 with round-to-nearest-even and saturation to +-448 for finite
 * values beyond range ("satfinite"); NaN -> NaN.  The magnitude is written as
 * a multiple of its binade's quantum (2^(E-3) for normal binades, 2^-9 below
 * 2^-6), rounded to the nearest even multiple; a rounding carry into the next
 * binade lands on the next code because codes are ordered like magnitudes. */
ORC_API uint8_t oracle_e4m3_from_f32(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;
    if (E < -6) {
        double m = rint(a / ldexp(1.0, -9)); /* 0 .. 8 */
        return (uint8_t)(sign | (int)m);
    }
    double m = rint(a / ldexp(1.0, E - 3)); /* 8 .. 16 */
    int code = ((E + 7) << 3) + ((int)m - 8);
    if (code > 0x7E)
        code = 0x7E;
    return (uint8_t)(sign | code);
}

/* The conversion above applied to an array (a loop over the scalar function). */
ORC_API void oracle_e4m3_from_f32_array(const float *x, size_t n, uint8_t *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_from_f32(x[i]);
}

/* Row-wise FP8 quantization of an N x D fp32 payload (p1 "Numeric Example" and
 * "Pinterest QComms Example": embedding lookup payloads go FP32 -> FP8 before
 * the collective).  Per row r (a reading: absmax scaling onto E4M3's range):
 *   a = max |x_rj| (+0)   sc = a / 448
 *   sc == 0 -> codes 0, row_scale = 0
 *   else code_rj = e4m3(x_rj / sc), row_scale = sc
 * Codes are row-major bytes; the fp32 scales are a separate array. */
ORC_API int oracle_rowwise_fp8(const float *x, size_t rows, size_t dim, uint8_t *codes,
                               float *row_scale)
{
    for (size_t r = 0; r < rows; ++r) {
        const float *xr = x + r * dim;
        float a = 0.0f;
        for (size_t j = 0; j < dim; ++j) {
            float v = fabsf(xr[j]);
            if (v > a)
                a = v;
        }
        a = orc_positive_zero(a);
        float sc = a / 448.0f;
        for (size_t j = 0; j < dim; ++j)
            codes[r * dim + j] = (sc == 0.0f) ? 0 : oracle_e4m3_from_f32(xr[j] / sc);
        row_scale[r] = sc;
    }
    return 0;
}

/* Receiver side of the FP8 payload: x_rj ~= e4m3_value(code_rj) * sc_r
 * (p1 "Where Quantization Sits": dequantize on receipt). */
ORC_API int oracle_rowwise_fp8_dequant(const uint8_t *codes, const float *row_scale, size_t rows,
                                       size_t dim, float *out)
{
    for (size_t r = 0; r < rows; ++r)
        for (size_t j = 0; j < dim; ++j)
            out[r * dim + j] = oracle_e4m3_to_f32(codes[r * dim + j]) * row_scale[r];
    return 0;
}
