/*
 * qcodec.h -- C ABI of libqcodec, the communication codec that wraps a collective
 * in data-parallel training: the sender quantizes a tensor for the wire, the
 * receiver dequantizes (and aggregates) what arrived.
 *
 * Sources, by page title and section:
 *   "Quantized Communication for Distributed Training", "Where Quantization Sits"
 *       (quantize for wire -> collective -> dequantize on receipt) and "Numeric
 *       Example" / "Pinterest QComms Example" (FP32 -> FP8 embedding payloads).
 *   "Quantization for Communication", "Quantization Schemes" (uniform min/max,
 *       stochastic rounding), "Quantized SGD Algorithms" (TernGrad, SignSGD with
 *       majority vote), "Error Feedback for Quantization", "Quantization-Aware
 *       All-Reduce" (accumulate in higher precision), "Hardware Acceleration"
 *       (several low-bit values packed per 32-bit word).
 *   "Gradient Compression and Quantised Collectives", "Why sparsification fights
 *       the all-reduce" (signSGD majority vote) and "Error feedback is the
 *       component that makes it work".
 *
 * Conventions shared by every call:
 *   - Every buffer pointer is a DEVICE pointer on the current CUDA device.  The
 *     caller allocates and frees every buffer; the library never allocates,
 *     frees, or synchronises, and keeps no device state between calls apart from
 *     the error flags that qc_take_device_errors() reads (and, per host
 *     thread, the status word address of qc_set_status_word).
 *   - Every compute call is asynchronous on `stream` (0 = legacy default stream).
 *     Arguments are validated on the host before any launch; on a non-OK status
 *     nothing was launched and nothing was written, and qc_last_error() holds a
 *     message.  QC_ERR_CUDA reports a launch error (cudaGetLastError after the
 *     launch); a fault inside a kernel surfaces at the caller's next
 *     synchronisation, as with any CUDA launch.
 *   - n == 0 (or rows == 0) is a valid no-op that returns QC_OK.
 *   - Outputs must not overlap inputs (checked for the buffers named per call).
 *   - Element i of a flat tensor belongs to bucket k = i / bucket; bucket k spans
 *     [k*bucket, min((k+1)*bucket, n)), so the last bucket may be partial.
 *   - Packed codes: code i of a b-bit stream sits in 32-bit word i / (32/b) at
 *     bit offset (i mod (32/b)) * b, least significant bits first.  Because
 *     bucket % 32 == 0 no word holds codes of two buckets.  Padding codes past n
 *     in the last word are written as 0.
 *   - Arithmetic is IEEE-754 binary32 with round-to-nearest-even, one rounding per
 *     operation as listed for each call; results are deterministic and do not
 *     depend on the launch shape.
 *   - Inputs are expected finite.  A NaN or infinity in a gradient never faults
 *     and never spills into another element's code: the codes of the non-finite
 *     elements (and, for the uniform scheme, their bucket's scale when the first
 *     element is one) are unspecified, the other elements' outputs are as stated.
 */
#ifndef QCODEC_H
#define QCODEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t. */
typedef struct CUstream_st *qc_stream_t;

typedef enum {
    QC_OK = 0,
    QC_ERR_NULL = 1,          /* a required pointer is NULL                        */
    QC_ERR_INVALID_ARG = 2,   /* bad size, bits, bucket, scheme, flag or overlap    */
    QC_ERR_ALIGNMENT = 3,     /* a pointer or stride breaks the stated alignment    */
    QC_ERR_UNSUPPORTED = 4,   /* valid in principle, outside the library's limits  */
    QC_ERR_CUDA = 5           /* the CUDA runtime reported an error at launch       */
} qc_status;

typedef enum {
    QC_SCHEME_UNIFORM = 0,    /* per-bucket min/max, 2^bits levels, fp32 scale+offset */
    QC_SCHEME_SIGN = 1,       /* 1 bit: sign, per-bucket fp32 scale = mean |p|        */
    QC_SCHEME_TERNARY = 2,    /* 2 bits: {-1,0,+1} -> codes {0,1,2}, scale = max |p|  */
    QC_SCHEME_QSGD = 3,       /* sign bit over bits-1 level bits, scale = ||p||_2 / s */
    QC_SCHEME_UNIFORM_CLIP = 4, /* uniform over the 1st..99th percentile range         */
    QC_SCHEME_LOG = 5         /* sign bit over a power-of-two level index, s = max |p| */
} qc_scheme;

typedef enum {
    QC_ROUND_NEAREST = 0,
    QC_ROUND_STOCHASTIC = 1   /* Philox4x32-10 keyed on (seed, step, element index) */
} qc_round;

typedef enum { QC_DTYPE_F32 = 0, QC_DTYPE_BF16 = 1 } qc_dtype;

enum {
    QC_OUT_SUM = 0,
    QC_OUT_MEAN = 1,                 /* divide the fixed-order sum by M             */
    QC_ACCUMULATE_INTO_OUT = 2       /* out = out + result instead of out = result  */
};

/* Largest supported worker count for decode and vote, and largest FP8 row. */
#define QC_MAX_WORKERS 1024
#define QC_MAX_FP8_DIM 4096

/* Number of 32-bit words holding n codes of `bits` bits: ceil(n*bits/32). */
size_t qc_code_words(size_t n, int bits);

/* Number of buckets of `bucket` elements covering n elements: ceil(n/bucket);
 * 0 when bucket is 0. */
size_t qc_num_buckets(size_t n, size_t bucket);

/*
 * qc_encode_ef -- sender half: error-feedback compression of one flat gradient.
 *
 * "Quantization for Communication", "Error Feedback for Quantization":
 *   e = e + grad; q = quantize(e); e = e - dequantize(q); communicate q.
 * With err == NULL there is no error feedback and p = grad.
 *
 * Per element:  p_i = fl(err_i + grad_i)    (bf16 grad is widened exactly)
 * Per bucket k, by scheme:
 *   UNIFORM ("Quantization Schemes"): mn = min p, mx = max p (a zero result is
 *     taken as +0), L = 2^bits - 1, scale = fl(fl(mx - mn) / L).
 *     scale == 0: q_i = 0.  Else t_i = fl(fl(p_i - mn) / scale) and
 *       NEAREST:    q_i = min(rint(t_i), L)                 (ties to even)
 *       STOCHASTIC: q_i = min(floor(t_i) + [u_i < t_i - floor(t_i)], L)
 *     deq_i = fma(q_i, scale, mn) (one rounding); scale[k] = scale, offset[k] = mn.
 *   SIGN ("Quantized SGD Algorithms", SignSGD; bits must be 1, mode NEAREST):
 *     s = mean over the bucket's elements of |p_i|, rounded once to binary32
 *     from a compensated (double-word) sum; bit_i = [p_i >= 0];
 *     deq_i = bit_i ? s : -s; scale[k] = s.  Within 1e-6 * max|p| of the exact
 *     mean (the sum's order of operations is the only freedom).
 *   TERNARY ("Quantized SGD Algorithms", TernGrad; bits must be 2):
 *     s = max |p| (+0 for an all-zero bucket, then every code is 1).
 *       STOCHASTIC: keep_i = [u_i < fl(|p_i| / s)];  NEAREST: keep_i = [fl(|p_i|/s) > 0.5]
 *     code_i = keep_i ? (p_i > 0 ? 2 : 0) : 1; deq_i = (code_i - 1) * s; scale[k] = s.
 *   QSGD ("Quantized SGD Algorithms", QSGD; bits 2, 4 or 8): s = 2^(bits-1) - 1,
 *     nrm = ||p||_2 over the bucket rounded to binary32, unit = fl(nrm / s).
 *     unit == 0: every code 0.  Else t_i = fl(|p_i| / unit) and the level is
 *       NEAREST:    l_i = min(rint(t_i), s)
 *       STOCHASTIC: l_i = min(floor(t_i) + [u_i < t_i - floor(t_i)], s)
 *     code_i = [p_i < 0] << (bits-1) | l_i; deq_i = +-fl(l_i * unit); scale[k] = unit.
 *     nrm is the binary32 value nearest (ties to even) to the square root of the
 *     EXACT sum of the squares (non-finite elements left out of the sum).
 *   UNIFORM_CLIP ("Adaptive Quantization Strategies", Percentile Clipping; bits
 *     1, 2, 4 or 8): as UNIFORM, but mn and mx are the bucket's nearest-rank 1st
 *     and 99th percentiles (the elements of 0-based rank ceil(cnt/100) - 1 and
 *     ceil(99 cnt/100) - 1 in sorted order; zero taken as +0), and every p_i is
 *     clamped into [mn, mx] before t_i is formed.  deq_i is that of the clamped
 *     element, so with error feedback err_i = fl(p_i - deq_i) keeps the clipped
 *     part.  Buckets of at most 99 elements reduce to UNIFORM.  Needs a bucket of
 *     at most 4096 elements and a 16-byte aligned gradient (else
 *     QC_ERR_UNSUPPORTED).  The payload decodes as UNIFORM.
 *   LOG ("Quantization Schemes", Non-Uniform Quantization: logarithmic levels,
 *     finer near zero; bits 2, 4 or 8): J = 2^(bits-1) - 1, s = max |p| (zero
 *     taken as +0), level magnitudes 0 (j = 0) and fl(s * 2^(j - J)) (j = 1..J).
 *     s == 0: every code 0.  Else x = fl(|p_i| / s) and
 *       x >= 1: j = J
 *       2^(1-J) <= x < 1: x = 2^e (1 + m), 0 <= m < 1 (exact), and
 *         NEAREST:    j = e + J + [m > 1/2, or m = 1/2 and e + J odd]
 *         STOCHASTIC: j = e + J + [u_i < m]
 *       x < 2^(1-J): f = x * 2^(J-1) (exact) and j = NEAREST ? [f > 1/2] : [u_i < f]
 *     code_i = [p_i < 0] << (bits-1) | j; deq_i = +-(j ? fl(s * 2^(j - J)) : 0);
 *     scale[k] = s.
 * Then, with error feedback, err_i = fl(p_i - deq_i) is written in place.
 *
 * Stochastic draw for element i (global index within this call):
 *   Philox4x32-10 (Salmon et al., SC'11) with key = (seed low 32, seed high 32),
 *   counter = (i/4 low 32, i/4 high 32, step, 0); u_i = (word (i mod 4) >> 8) * 2^-24.
 *
 * grad   : n elements of `dtype`; 16-byte aligned (f32) or 8-byte aligned (bf16).
 * err    : n fp32, in/out, 16-byte aligned, or NULL for no error feedback.
 * bits   : UNIFORM and UNIFORM_CLIP 1, 2, 4 or 8; SIGN 1; TERNARY 2; QSGD and LOG
 *          2, 4 or 8.
 * bucket : elements per bucket, a multiple of 32, 32 <= bucket <= 2^24.
 * codes  : out, qc_code_words(n, bits) uint32 words, 4-byte aligned.
 * scale  : out, qc_num_buckets(n, bucket) fp32.
 * offset : out, qc_num_buckets(n, bucket) fp32 for UNIFORM and UNIFORM_CLIP;
 *          ignored otherwise (may be NULL).
 */
qc_status qc_encode_ef(const void *grad, qc_dtype dtype, float *err, size_t n, int bits,
                       size_t bucket, qc_scheme scheme, qc_round mode, uint64_t seed,
                       uint32_t step, uint32_t *codes, float *scale, float *offset,
                       qc_stream_t stream);

/*
 * qc_encode_ef_segments -- qc_encode_ef over a list of flat gradients in one
 * launch (or one per QC_MAX_SEGMENTS_PER_LAUNCH segments).
 *
 * "Gradient Compression and Quantised Collectives", "When it breaks": small
 * tensors make the launch cost dominate, and bucketing many small tensors into
 * one exchange is what makes the all-reduce efficient.  Here the tensors stay
 * where they are: each segment keeps its own arrays and its buckets start at
 * its own element 0, exactly as a separate qc_encode_ef call on it would, and
 * every output is that call's, bit for bit, except for the stochastic draws:
 * element i of segment s draws with the index I_s + i under the call's one seed
 * and step, where I_s = the sum over the segments r before s of n_r rounded up
 * to a multiple of 4.  That is the place of segment s when the segments are
 * laid end to end, each padded to a whole Philox block of four draws (16 bytes
 * of fp32), the way tensors are padded into a flat communication bucket; where
 * every n is a multiple of 4 the draws are those of one call over the
 * concatenation.  With one segment this is qc_encode_ef.
 *
 * segs   : nseg host-memory descriptors (nseg == 0 is a no-op); a segment with
 *          n == 0 is skipped.  Every field is as for qc_encode_ef's argument of
 *          the same name; err must be given for every segment or for none.
 *          No output of a segment may overlap any buffer of another segment.
 * dtype, bits, bucket, scheme, mode, seed, step : as for qc_encode_ef, shared by
 *          every segment.
 * One launch covers the segments when every one suits the same kernel: the
 * receiver's bf16 encode (8-bit nearest or ternary stochastic, no residual,
 * buckets of 1024) or the pipelined encode (16-byte aligned gradients, buckets
 * of at most 4096 elements, any scheme but UNIFORM_CLIP); otherwise each
 * segment takes its own launch, with the same results.  Validation of every
 * segment precedes every launch.
 */
typedef struct {
    const void *grad;   /* n elements of the call's dtype                          */
    float *err;         /* n fp32 residual (in/out), or NULL                        */
    size_t n;           /* elements                                                 */
    uint32_t *codes;    /* out: qc_code_words(n, bits) words                        */
    float *scale;       /* out: qc_num_buckets(n, bucket)                           */
    float *offset;      /* out: qc_num_buckets(n, bucket) (uniform schemes), or NULL */
} qc_segment;

#define QC_MAX_SEGMENTS_PER_LAUNCH 60

qc_status qc_encode_ef_segments(const qc_segment *segs, int nseg, qc_dtype dtype, int bits,
                                size_t bucket, qc_scheme scheme, qc_round mode, uint64_t seed,
                                uint32_t step, qc_stream_t stream);

/*
 * qc_decode_accumulate -- receiver half: dequantize M workers' payloads and
 * accumulate them in fp32.
 *
 * "Quantization for Communication", "Quantization-Aware All-Reduce" (dequantize
 * after the exchange; accumulate in higher precision) and "Gradient quantization
 * for communication", "How Gradient Quantization Works" (dequantize, then
 * average or sum).  For every element i (bucket k = i / bucket):
 *   acc = +0; for w = 0 .. M-1 in this order: acc = fl(acc + d_w,i) with
 *     UNIFORM d = fma(q, scale_w[k], offset_w[k]); SIGN d = bit ? s_w[k] : -s_w[k];
 *     TERNARY d = (code - 1) * s_w[k]; QSGD d = +-fl(level * unit_w[k]) with the
 *     sign from the code's top bit and the level from the rest; LOG
 *     d = +-(j ? fl(s_w[k] * 2^(j - J)) : 0), the sign (a zero level keeps it,
 *     giving -0) from the top bit and j from the rest
 *   r = (flags & QC_OUT_MEAN) ? fl(acc / M) : acc
 *   out_i = (flags & QC_ACCUMULATE_INTO_OUT) ? fl(out_i + r) : r
 *
 * codes  : worker w's packed codes start at codes + w * codes_stride_words
 *          (codes_stride_words >= qc_code_words(n, bits) when M > 1); 4-byte aligned.
 * scale  : worker w's per-bucket scales at scale + w * meta_stride
 *          (meta_stride >= qc_num_buckets(n, bucket) when M > 1).
 * offset : same layout as scale; UNIFORM and UNIFORM_CLIP only (ignored
 *          otherwise, may be NULL).
 * M      : 1 .. QC_MAX_WORKERS.   bits/scheme as for qc_encode_ef (an
 *          UNIFORM_CLIP payload decodes exactly as a UNIFORM one).
 * out    : n fp32, 16-byte aligned; read only with QC_ACCUMULATE_INTO_OUT.
 */
qc_status qc_decode_accumulate(const uint32_t *codes, size_t codes_stride_words,
                               const float *scale, const float *offset, size_t meta_stride,
                               int M, size_t n, int bits, size_t bucket, qc_scheme scheme,
                               float *out, int flags, qc_stream_t stream);

/*
 * qc_reencode -- receiver re-encode: the far side of a two-phase quantized
 * all-reduce.  The owner of a shard decodes the M workers' payloads of that
 * shard, accumulates them, and quantizes the result again, with its own
 * error-feedback residual, for the all-gather phase ("Quantization for
 * Communication", "Quantization-Aware All-Reduce": dequantize after the
 * exchange, accumulate in higher precision; "Gradient Compression and
 * Quantised Collectives": reduce-scatter then all-gather).  Per element:
 *   r_i = qc_decode_accumulate's result with `flags` (QC_OUT_SUM or QC_OUT_MEAN;
 *         QC_ACCUMULATE_INTO_OUT is not accepted)
 *   then qc_encode_ef of r (as an F32 gradient) with residual `err`, the SAME
 *   scheme, bits and bucket as the incoming payloads, `mode`, `seed`, `step`:
 *   p_i = err ? fl(err_i + r_i) : r_i, the scheme's statistics, codes and,
 *   with err, err_i = fl(p_i - deq_i).
 * The result equals qc_decode_accumulate into a buffer followed by qc_encode_ef
 * of that buffer, bit for bit; one kernel does both without the fp32 round trip.
 *
 * codes, scale, offset, meta_stride, codes_stride_words, M, bits, bucket,
 * scheme : as for qc_decode_accumulate (UNIFORM_CLIP: QC_ERR_UNSUPPORTED, the
 *          clipped encode is not fused here).  `codes` must be 16-byte aligned and,
 *          for M > 1, codes_stride_words a multiple of 4, and the bucket at
 *          most 8192 elements; otherwise QC_ERR_UNSUPPORTED (the two-call
 *          composition above serves those layouts).
 * err    : n fp32 residual of this receiver, in/out, 16-byte aligned, or NULL.
 * mode, seed, step : as for qc_encode_ef (SIGN needs NEAREST).
 * codes_out, scale_out, offset_out : the new payload, laid out as
 *          qc_encode_ef's outputs (offset_out UNIFORM only, else may be NULL).
 * out    : n fp32, 16-byte aligned, receives r; or NULL to skip it.
 * No output may overlap an input or another output.
 */
qc_status qc_reencode(const uint32_t *codes, size_t codes_stride_words, const float *scale,
                      const float *offset, size_t meta_stride, int M, size_t n, int bits,
                      size_t bucket, qc_scheme scheme, int flags, float *err, qc_round mode,
                      uint64_t seed, uint32_t step, uint32_t *codes_out, float *scale_out,
                      float *offset_out, float *out, qc_stream_t stream);

/*
 * qc_topk_encode_ef -- top-k sparsification with 8-bit codes and error feedback
 * ("Gradient quantization for communication", "Quantization Schemes": send only
 * the largest K% of gradients, combined with quantization, with error
 * feedback; "Quantization for Communication", "Combination with Other
 * Techniques"; "Gradient Compression and Quantised Collectives", "Why
 * sparsification fights the all-reduce": the exchange is index-value pairs).
 * Per bucket k of cnt elements, K = min(keep, cnt):
 *   p_i = err ? fl(err_i + grad_i) : grad_i
 *   kept = the K elements of largest |p_i|, ties to the lower index
 *   mn, mx = min and max of p over kept (zero taken as +0); scale = fl(fl(mx-mn)/255)
 *   each kept element: q_i and deq_i exactly as qc_encode_ef's UNIFORM 8-bit
 *     (NEAREST or STOCHASTIC, the draw of element i)
 *   err_i = kept ? fl(p_i - deq_i) : p_i
 * Slot t (0 <= t < keep) of bucket k, at k*keep + t: the t-th kept element in
 * ascending index order, idx = its index (0-based in this call), codes = q;
 * slots t >= K (a short last bucket) hold idx 0xFFFFFFFF and code 0.
 * scale[k] = scale, offset[k] = mn.
 *
 * grad   : n elements of `dtype`, 16-byte aligned (else QC_ERR_UNSUPPORTED).
 * err    : n fp32, in/out, 16-byte aligned, or NULL for no error feedback.
 * bucket : a multiple of 32, at most 4096 (else QC_ERR_UNSUPPORTED).
 * keep   : kept elements per bucket, 1 .. bucket.
 * idx    : out, qc_num_buckets(n, bucket) * keep uint32.
 * codes  : out, qc_num_buckets(n, bucket) * keep bytes.
 * scale, offset : out, qc_num_buckets(n, bucket) fp32 each.
 * n must be below 2^32 (32-bit indices).
 */
qc_status qc_topk_encode_ef(const void *grad, qc_dtype dtype, float *err, size_t n, size_t bucket,
                            uint32_t keep, qc_round mode, uint64_t seed, uint32_t step,
                            uint32_t *idx, uint8_t *codes, float *scale, float *offset,
                            qc_stream_t stream);

/*
 * qc_topk_decode_accumulate -- receiver of top-k payloads: the M workers' pairs
 * scattered into a dense fp32 vector and accumulated in fixed worker order.
 *   acc_i = +0; for w = 0 .. M-1, for every bucket k and slot t:
 *     i = idx_w[k*keep + t]; skipped unless k*bucket <= i < min((k+1)*bucket, n)
 *     acc_i = fl(acc_i + fma(code, scale_w[k], offset_w[k]))
 *   r = (flags & QC_OUT_MEAN) ? fl(acc / M) : acc
 *   out_i = (flags & QC_ACCUMULATE_INTO_OUT) ? fl(out_i + r) : r
 * A worker's indices within one bucket must be distinct (as the encoder writes
 * them); duplicates leave that element's sum unspecified (never out of bounds).
 *
 * idx, codes : worker w's slots start at w * pair_stride
 *              (pair_stride >= qc_num_buckets(n, bucket) * keep when M > 1).
 * scale, offset : worker w's at w * meta_stride (>= qc_num_buckets when M > 1).
 * M      : 1 .. QC_MAX_WORKERS.  bucket <= 16384, keep <= 1024 (else
 *          QC_ERR_UNSUPPORTED).  out : n fp32, 4-byte aligned.
 */
qc_status qc_topk_decode_accumulate(const uint32_t *idx, const uint8_t *codes, size_t pair_stride,
                                    const float *scale, const float *offset, size_t meta_stride,
                                    int M, size_t n, size_t bucket, uint32_t keep, float *out,
                                    int flags, qc_stream_t stream);

/*
 * qc_sign_vote -- signSGD aggregation by majority vote ("Quantization for
 * Communication", "Quantized SGD Algorithms"; "Gradient Compression and
 * Quantised Collectives", "Why sparsification fights the all-reduce").
 *   c_i = number of workers whose sign bit i is set;  out bit i = [2 * c_i >= M]
 * (a tie, possible for even M, gives 1, matching sign(0) = +1).  Bits past n in
 * the last word are written as 0.
 *
 * signs        : worker w's qc_code_words(n, 1) words at signs + w * stride_words,
 *                stride_words >= qc_code_words(n, 1) when M > 1; 4-byte aligned.
 * M            : 1 .. QC_MAX_WORKERS.
 * out          : qc_code_words(n, 1) uint32, 4-byte aligned.
 * The vectorised path is taken when signs, out and stride_words keep 16-byte
 * alignment; otherwise a word-at-a-time path gives the same result.
 */
qc_status qc_sign_vote(const uint32_t *signs, size_t stride_words, int M, size_t n,
                       uint32_t *out, qc_stream_t stream);

/*
 * qc_rowwise_fp8 -- FP32 -> FP8 (OCP E4M3) row-wise quantization of an
 * embedding lookup payload ("Quantized Communication for Distributed Training",
 * "Numeric Example" and "Pinterest QComms Example").  Per row r:
 *   a = max_j |x_rj| (+0 if zero);  sc = fl(a / 448)
 *   sc == 0: codes 0x00, row_scale = 0;  else code_rj = e4m3_rn_satfinite(fl(x_rj / sc))
 * x         : rows x dim fp32, row-major, 16-byte aligned.
 * dim       : a multiple of 4, 4 <= dim <= QC_MAX_FP8_DIM.
 * codes     : out, rows x dim bytes, row-major, 4-byte aligned.
 * row_scale : out, rows fp32.
 */
qc_status qc_rowwise_fp8(const float *x, size_t rows, size_t dim, uint8_t *codes,
                         float *row_scale, qc_stream_t stream);

/*
 * qc_rowwise_fp8_dequant -- receiver side of the FP8 payload:
 *   out_rj = fl(e4m3_value(code_rj) * row_scale_r)   (the e4m3 value is exact)
 * Layouts and limits as for qc_rowwise_fp8; out is 16-byte aligned.
 */
qc_status qc_rowwise_fp8_dequant(const uint8_t *codes, const float *row_scale, size_t rows,
                                 size_t dim, float *out, qc_stream_t stream);

/*
 * qc_take_device_errors -- device-side failures of the pipelined kernels.
 *
 * The kernels that stream tiles through shared memory wait on mbarriers for at
 * most 2 s (of the GPU's global timer, and of its SM cycle counter); a wait that runs out stops its block and
 * sets a flag in device memory instead of spinning forever.  This call
 * synchronises the current device, stores the OR of the flags set since the
 * previous call in *flags (bit 0: a pipeline wait timed out; the outputs of
 * that launch are incomplete: the tiles whose wait timed out, and the ones after
 * them in that block, are not written, so an encode's residual keeps its old
 * values there) and clears them, each flag in one atomic
 * exchange, so a flag set concurrently is reported by this call or the next,
 * never lost.  A CUDA error while reading them returns QC_ERR_CUDA.  It is a
 * diagnostic call: it blocks the host and must not be used inside stream
 * capture.  qc_set_status_word gives the same information per launch, in
 * stream order, without a synchronisation.
 */
qc_status qc_take_device_errors(uint32_t *flags);

/*
 * qc_set_status_word -- per-launch failure reporting in stream order.
 *
 * Every launch that the library issues from the calling host thread after this
 * call carries `status` (a device address of one 32-bit word; NULL turns it
 * off): if the launch's bounded waits run out, the kernel ORs the failure bits
 * (bit 0: a pipeline wait timed out) into *status as well as into the flags of
 * qc_take_device_errors.  The caller zeroes the word (for example with
 * cudaMemsetAsync) before the launches it wants to watch and reads it back on
 * the same stream after them; no synchronisation of the device is needed.  The
 * word must stay valid until those launches have run.  Only the kernels that
 * wait on a pipeline can fail this way; the others never write the word.
 * status must be 4-byte aligned (else QC_ERR_ALIGNMENT).  The setting is
 * per host thread and lasts until the next call.
 */
qc_status qc_set_status_word(uint32_t *status);

/*
 * qc_selftest_wait_timeout -- exercises the failure path that
 * qc_take_device_errors() and the status word report, without a fault: one
 * block waits on a shared-memory barrier that nothing completes, with the
 * pipelines' time-bounded wait limited to `timeout_us` microseconds
 * (1 .. 10^7, else QC_ERR_INVALID_ARG).  The wait runs out, the block sets the
 * pipeline-timeout flag (bit 0), and the status word if one is set, and
 * returns; the context stays usable.  Asynchronous on `stream`.
 */
qc_status qc_selftest_wait_timeout(uint32_t timeout_us, qc_stream_t stream);

/* Message for the last non-OK status returned on the calling thread ("" if none). */
const char *qc_last_error(void);

/* Library version string. */
const char *qc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QCODEC_H */
