// qc_api.cu -- the C ABI of libqcodec (declared in include/qcodec.h): host-side
// validation, dispatch to the kernels, and error reporting.  Validation touches
// no CUDA API, so every argument error is reported without any device work.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <algorithm>
#include <map>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/qcodec.h"
#include "qc_internal.h"

static_assert(int{QC_SCHEME_UNIFORM} == qc::kUniform && int{QC_SCHEME_SIGN} == qc::kSign &&
                  int{QC_SCHEME_TERNARY} == qc::kTernary && int{QC_SCHEME_QSGD} == qc::kQsgd &&
                  int{QC_SCHEME_UNIFORM_CLIP} == qc::kClip && int{QC_SCHEME_LOG} == qc::kLog,
              "the public scheme numbers are the kernels' template arguments");
static_assert(QC_MAX_SEGMENTS_PER_LAUNCH == qc::kMaxSegments, "one segment table per launch");

namespace {

thread_local char g_last_error[512] = "";
// The status word that launches from this thread report failures into.
thread_local uint32_t *g_status_word = nullptr;

qc_status fail(qc_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

qc_status ok() {
    g_last_error[0] = '\0';
    return QC_OK;
}

qc_status from_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return ok();
    return fail(QC_ERR_CUDA, "%s: CUDA error %d (%s)", what, static_cast<int>(e),
                cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [a, a+na) and [b, b+nb) (bytes) share a byte.
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool valid_bucket(size_t bucket) { return bucket >= 32 && bucket % 32 == 0 && bucket <= (1u << 24); }

// Team of W warps per bucket: the smallest power of two with 512 W >= bucket,
// capped at the 8 warps of a block (larger buckets take two passes).
int team_warps_for(size_t elems) {
    int w = 1;
    while (w < 8 && static_cast<size_t>(qc::kWindowPerWarp) * w < elems) w <<= 1;
    return w;
}

// Tiling for the TMA-pipelined encode: whole buckets per tile, the bucket count
// a multiple of the block's teams, at least 16 KB of input per stage.  Stages
// under 32 KB come three to a block (room for 4 blocks per SM); from 32 KB on
// two, so that three blocks share an SM (measured 2-16 % faster for the fp32
// encodes with error feedback), except that a block of one team (4096-element
// buckets) keeps three 32 KB stages, which measured faster there.  Buckets
// larger than one team window (4096) and gradients whose base is not 16-byte
// aligned take the direct kernel.
bool encode_tiles_for(const qc::EncodeParams &p, size_t esize, bool ef, bool grad16,
                      qc::EncodeTiles &t, size_t extra_smem = 0) {
    if (!grad16 || p.two_pass) return false;
    const size_t per_elem = esize + (ef ? 4 : 0);
    const uint32_t teams = (qc::kBlock / 32) / p.team_warps;
    const size_t target = 16 * 1024;
    uint32_t tb = static_cast<uint32_t>(target / (static_cast<size_t>(p.bucket) * per_elem));
    tb = tb / teams * teams;
    if (tb < teams) tb = teams;
    const size_t stage = static_cast<size_t>(tb) * p.bucket * per_elem;
    if (stage > 64 * 1024) return false;
    uint32_t stages = (stage < 32 * 1024 || (stage == 32 * 1024 && teams == 1)) ? 3u : 2u;
    // kernels with per-team selection buffers keep two blocks per SM
    if (stages == 3 && 3 * stage + extra_smem > 110 * 1024) stages = 2;
    t.tb = tb;
    t.te = tb * p.bucket;
    t.stages = stages;
    t.stage_bytes = static_cast<uint32_t>(stage);
    t.e_offset = static_cast<uint32_t>(static_cast<size_t>(t.te) * esize);
    t.ntiles = (p.n + t.te - 1) / t.te;
    return true;
}

// Tiling for the bf16 encode without error feedback: buckets of 1024, 2048,
// 4096 or 8192 elements, W = bucket / 1024 warps per bucket, whole buckets per
// tile, about 16 KB of bf16 per stage, three stages.
bool bf16_tiles_for(const qc::EncodeParams &p, bool grad16, qc::EncodeTiles &t) {
    if (!grad16 || p.err != nullptr || p.bucket > 8192) return false;
    uint32_t w = 1;
    while (w < 8 && 1024u * w < p.bucket) w <<= 1;
    // a team covers exactly one bucket (1024 elements per warp); other bucket
    // sizes take the general pipelined kernel
    if (p.bucket != 1024u * w) return false;
    const uint32_t teams = (qc::kBlock / 32) / w;
    uint32_t tb = static_cast<uint32_t>((16 * 1024) / (static_cast<size_t>(p.bucket) * 2));
    tb = tb / teams * teams;
    if (tb < teams) tb = teams;
    t.warps = w;
    t.tb = tb;
    t.te = tb * p.bucket;
    t.stage_bytes = t.te * 2;
    t.stages = t.stage_bytes <= 32 * 1024 ? 3u : 2u;
    t.e_offset = 0;
    t.ntiles = (p.n + t.te - 1) / t.te;
    return true;
}

uint64_t gcd_u64(uint64_t a, uint64_t b) {
    while (b) {
        const uint64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Tiling for the pipelined decode: tiles of whole buckets whose element count
// is a multiple of 128 (so every worker's code slice starts on a 16-byte
// boundary), about 32 KB of codes per stage, three stages.  Payloads whose
// worker stride or base breaks 16-byte alignment, and worker counts whose
// smallest tile does not fit, take the direct kernel.
bool decode_tiles_for(const qc::DecodeParams &p, int bits, qc::DecodeTiles &t) {
    // Few workers: the decode is dominated by its fp32 stores, which the direct
    // kernel's higher occupancy serves better.
    if (p.M < 4) return false;
    if (!aligned(p.codes, 16) || p.codes_stride % 4 != 0) return false;
    const uint64_t unit = static_cast<uint64_t>(p.bucket) / gcd_u64(p.bucket, 128) * 128;
    const uint64_t bytes_per_elem_x8 = static_cast<uint64_t>(p.M) * bits;  // code bits per element
    // 2-bit payloads take half-size stages, four of them, so that three blocks
    // share an SM (their consumers are the shorter-latency part of the kernel)
    const uint64_t target = bits <= 2 ? 16 * 1024 : 32 * 1024;
    uint64_t te = (target * 8 / bytes_per_elem_x8) / unit * unit;
    if (te < unit) te = unit;
    const uint64_t worker_bytes = te * bits / 8;
    const uint64_t tb = te / p.bucket;
    const uint64_t meta_bytes = 8 * static_cast<uint64_t>(p.M) * tb;
    const uint64_t stage = (static_cast<uint64_t>(p.M) * worker_bytes + meta_bytes + 127) / 128 * 128;
    if (stage > 64 * 1024 || te > (1u << 30)) return false;
    t.tb = static_cast<uint32_t>(tb);
    t.te = static_cast<uint32_t>(te);
    t.worker_bytes = static_cast<uint32_t>(worker_bytes);
    t.meta_offset = static_cast<uint32_t>(p.M * worker_bytes);
    t.stage_bytes = static_cast<uint32_t>(stage);
    t.stages = stage <= 18 * 1024 ? 4u : stage <= 36 * 1024 ? 3u : 2u;
    int sh = -1;
    if ((p.bucket & (p.bucket - 1)) == 0) {
        sh = 0;
        while ((1u << sh) < p.bucket) ++sh;
    }
    t.bucket_shift = sh;
    t.ntiles = (p.n + te - 1) / te;
    return true;
}

// Tiling for the fused re-encode: tiles of whole buckets whose element count is
// a multiple of 128, 4096 elements where the bucket allows (one bucket when
// buckets are larger), so that both phases keep every consumer thread busy (16
// outputs per thread in the decode, a full set of teams in the encode); as many
// workers per stage as fit in about 26 KB of codes and metadata, the rest in
// further chunks, three stages.  Buckets above 8192 elements and payloads
// without 16-byte aligned worker slices are not supported.
bool reencode_tiles_for(const qc::ReencodeParams &p, int bits, qc::ReencodeTiles &t) {
    if (!aligned(p.codes, 16) || p.codes_stride % 4 != 0) return false;
    const uint64_t B = p.bucket;
    const uint64_t unit = B / gcd_u64(B, 128) * 128;
    if (unit > 8192) return false;
    const uint64_t budget = 26 * 1024;
    const uint64_t M = static_cast<uint64_t>(p.M);
    const uint64_t te = unit > 4096 ? unit : 4096 / unit * unit;
    const uint64_t worker_bytes = te * bits / 8;
    const uint64_t tb = te / B;
    const uint64_t per_worker = worker_bytes + 8 * tb;
    uint64_t mc = budget / per_worker;
    if (mc < 1) mc = 1;
    if (mc > M) mc = M;
    const uint64_t nchunks = (M + mc - 1) / mc;
    mc = (M + nchunks - 1) / nchunks;
    const uint64_t stage = (mc * per_worker + 127) / 128 * 128;
    t.tb = static_cast<uint32_t>(tb);
    t.te = static_cast<uint32_t>(te);
    t.mc = static_cast<uint32_t>(mc);
    t.nchunks = static_cast<uint32_t>(nchunks);
    t.worker_bytes = static_cast<uint32_t>(worker_bytes);
    t.meta_offset = static_cast<uint32_t>(mc * worker_bytes);
    t.stage_bytes = static_cast<uint32_t>(stage);
    t.stages = stage <= 28 * 1024 ? 3u : 2u;
    int sh = -1;
    if ((B & (B - 1)) == 0) {
        sh = 0;
        while ((1ull << sh) < B) ++sh;
    }
    t.bucket_shift = sh;
    t.ntiles = (p.n + te - 1) / te;
    return true;
}

// Bits and rounding mode allowed for a scheme; QC_OK or the failure status.
qc_status check_scheme(const char *fn, qc_scheme scheme, int bits) {
    if (scheme == QC_SCHEME_UNIFORM || scheme == QC_SCHEME_UNIFORM_CLIP) {
        if (bits != 1 && bits != 2 && bits != 4 && bits != 8)
            return fail(QC_ERR_INVALID_ARG, "%s: uniform bits must be 1, 2, 4 or 8 (got %d)", fn, bits);
    } else if (scheme == QC_SCHEME_SIGN) {
        if (bits != 1) return fail(QC_ERR_INVALID_ARG, "%s: sign scheme needs bits == 1 (got %d)", fn, bits);
    } else if (scheme == QC_SCHEME_TERNARY) {
        if (bits != 2) return fail(QC_ERR_INVALID_ARG, "%s: ternary scheme needs bits == 2 (got %d)", fn, bits);
    } else if (scheme == QC_SCHEME_QSGD) {
        if (bits != 2 && bits != 4 && bits != 8)
            return fail(QC_ERR_INVALID_ARG, "%s: QSGD bits must be 2, 4 or 8 (got %d)", fn, bits);
    } else if (scheme == QC_SCHEME_LOG) {
        if (bits != 2 && bits != 4 && bits != 8)
            return fail(QC_ERR_INVALID_ARG, "%s: logarithmic-level bits must be 2, 4 or 8 (got %d)", fn, bits);
    } else {
        return fail(QC_ERR_INVALID_ARG, "%s: unknown scheme %d", fn, scheme);
    }
    return QC_OK;
}

}  // namespace

namespace qc {

int persistent_grid(const void *kernel, int block, uint64_t units, size_t smem) {
    static std::mutex mu;
    // (device, kernel, block size, smem) -> blocks per SM
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    static std::unordered_map<int, int> sms;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, kernel, block, smem);
    int per_sm = 0, nsm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it == cache.end()) {
            int b = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, block, smem) != cudaSuccess ||
                b < 1)
                b = 1;
            it = cache.emplace(key, b).first;
        }
        per_sm = it->second;
        auto is = sms.find(dev);
        if (is == sms.end()) {
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
                n = 1;
            is = sms.emplace(dev, n).first;
        }
        nsm = is->second;
    }
    const uint64_t cap = static_cast<uint64_t>(per_sm) * static_cast<uint64_t>(nsm);
    uint64_t g = units < cap ? units : cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

cudaError_t prepare_dynamic_smem(const void *kernel, size_t bytes) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, size_t> done;  // (device, kernel) -> limit set
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t key = (static_cast<uint64_t>(dev) << 56) ^ reinterpret_cast<uintptr_t>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    // Prefer the largest shared-memory carveout so that several pipelined
    // blocks fit on one SM.
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done[key] = bytes;
    return e;
}

}  // namespace qc

extern "C" {

size_t qc_code_words(size_t n, int bits) {
    if (bits <= 0) return 0;
    return (n * static_cast<size_t>(bits) + 31) / 32;
}

size_t qc_num_buckets(size_t n, size_t bucket) {
    if (bucket == 0) return 0;
    return (n + bucket - 1) / bucket;
}

const char *qc_last_error(void) { return g_last_error; }

const char *qc_version(void) { return "libqcodec 0.2.0 (sm_103a)"; }

qc_status qc_set_status_word(uint32_t *status) {
    if (status && !aligned(status, 4))
        return fail(QC_ERR_ALIGNMENT, "qc_set_status_word: the status word must be 4-byte aligned");
    g_status_word = status;
    return ok();
}

qc_status qc_selftest_wait_timeout(uint32_t timeout_us, qc_stream_t stream) {
    if (timeout_us < 1 || timeout_us > 10000000u)
        return fail(QC_ERR_INVALID_ARG, "qc_selftest_wait_timeout: timeout_us must be in [1, 10^7] (got %u)",
                    timeout_us);
    return from_cuda(qc::launch_wait_timeout_selftest(timeout_us, g_status_word,
                                                      reinterpret_cast<cudaStream_t>(stream)),
                     "qc_selftest_wait_timeout");
}

qc_status qc_take_device_errors(uint32_t *flags) {
    if (!flags) return fail(QC_ERR_NULL, "qc_take_device_errors: flags must be non-NULL");
    *flags = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e, "qc_take_device_errors");
    cudaError_t (*const takes[])(uint32_t *) = {
        qc::take_encode_errors,          qc::take_encode_clip_errors, qc::take_encode_clip_bf16_errors,
        qc::take_reencode_other_errors,  qc::take_encode_log_errors,  qc::take_reencode_log_errors,
        qc::take_selftest_errors,        qc::take_topk_errors,        qc::take_encode_bf16_errors,
        qc::take_encode_bf16_fast_errors, qc::take_decode_errors,     qc::take_reencode_errors};
    uint32_t all = 0;
    for (auto take : takes) {
        uint32_t v = 0;
        e = take(&v);
        if (e != cudaSuccess) return from_cuda(e, "qc_take_device_errors");
        all |= v;
    }
    *flags = all;
    return ok();
}

}  // extern "C"

namespace {

// The call-wide arguments of an encode: QC_OK or the failure status.
qc_status check_encode_args(const char *fn, qc_dtype dtype, int bits, size_t bucket,
                            qc_scheme scheme, qc_round mode) {
    if (dtype != QC_DTYPE_F32 && dtype != QC_DTYPE_BF16)
        return fail(QC_ERR_INVALID_ARG, "%s: dtype %d is not F32 or BF16", fn, dtype);
    const qc_status sc = check_scheme(fn, scheme, bits);
    if (sc != QC_OK) return sc;
    if (scheme == QC_SCHEME_SIGN && mode != QC_ROUND_NEAREST)
        return fail(QC_ERR_INVALID_ARG, "%s: sign scheme is deterministic; mode must be NEAREST", fn);
    if (mode != QC_ROUND_NEAREST && mode != QC_ROUND_STOCHASTIC)
        return fail(QC_ERR_INVALID_ARG, "%s: unknown rounding mode %d", fn, mode);
    if (!valid_bucket(bucket))
        return fail(QC_ERR_INVALID_ARG, "%s: bucket must be a multiple of 32 in [32, 2^24] (got %zu)",
                    fn, bucket);
    return QC_OK;
}

// The buffers of one flat gradient (n > 0): pointers, alignment, overlaps.
qc_status check_encode_buffers(const char *fn, const void *grad, qc_dtype dtype, const float *err,
                               size_t n, int bits, size_t bucket, qc_scheme scheme,
                               const uint32_t *codes, const float *scale, const float *offset) {
    if (n > (static_cast<size_t>(1) << 40))
        return fail(QC_ERR_UNSUPPORTED, "%s: n = %zu exceeds 2^40 elements", fn, n);
    if (!grad || !codes || !scale) return fail(QC_ERR_NULL, "%s: grad, codes and scale must be non-NULL", fn);
    const bool uni = scheme == QC_SCHEME_UNIFORM || scheme == QC_SCHEME_UNIFORM_CLIP;
    if (uni && !offset) return fail(QC_ERR_NULL, "%s: the uniform schemes need an offset array", fn);
    const size_t esize = dtype == QC_DTYPE_F32 ? 4 : 2;
    if (!aligned(grad, dtype == QC_DTYPE_F32 ? 16 : 8))
        return fail(QC_ERR_ALIGNMENT, "%s: grad must be %d-byte aligned", fn, dtype == QC_DTYPE_F32 ? 16 : 8);
    if (err && !aligned(err, 16)) return fail(QC_ERR_ALIGNMENT, "%s: err must be 16-byte aligned", fn);
    if (!aligned(codes, 4) || !aligned(scale, 4) || (offset && !aligned(offset, 4)))
        return fail(QC_ERR_ALIGNMENT, "%s: codes, scale and offset must be 4-byte aligned", fn);
    const size_t nb = qc_num_buckets(n, bucket);
    const size_t cbytes = qc_code_words(n, bits) * 4, mbytes = nb * 4;
    const void *outs[3] = {codes, scale, uni ? offset : nullptr};
    const size_t osz[3] = {cbytes, mbytes, mbytes};
    for (int a = 0; a < 3; ++a) {
        if (overlaps(outs[a], osz[a], grad, n * esize) || overlaps(outs[a], osz[a], err, n * 4))
            return fail(QC_ERR_INVALID_ARG, "%s: an output overlaps grad or err", fn);
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], osz[a], outs[b], osz[b]))
                return fail(QC_ERR_INVALID_ARG, "%s: outputs overlap each other", fn);
    }
    if (overlaps(err, n * 4, grad, n * esize)) return fail(QC_ERR_INVALID_ARG, "%s: err overlaps grad", fn);
    return QC_OK;
}

// The call-wide part of the kernel parameters (the per-array fields are the
// caller's to fill).
qc::EncodeParams encode_params(size_t bucket, uint64_t seed, uint32_t step) {
    qc::EncodeParams p{};
    p.bucket = static_cast<uint32_t>(bucket);
    p.team_warps = team_warps_for(bucket);
    p.two_pass = bucket > static_cast<size_t>(qc::kWindowPerWarp) * p.team_warps ? 1 : 0;
    p.seed = seed;
    p.step = step;
    p.keys = qc::philox_round_keys(seed);
    p.status = g_status_word;
    return p;
}

// One flat gradient (validated), on the kernel its layout suits.
qc_status encode_one(const char *fn, const qc::EncodeParams &p, qc_dtype dtype, int bits,
                     qc_scheme scheme, qc_round mode, cudaStream_t st) {
    const size_t esize = dtype == QC_DTYPE_F32 ? 4 : 2;
    const bool grad16 = aligned(p.grad, 16), sr = mode == QC_ROUND_STOCHASTIC;
    const bool bf16 = dtype == QC_DTYPE_BF16;
    qc::EncodeTiles tiles{};
    if (scheme == QC_SCHEME_UNIFORM_CLIP) {
        // the percentile selection runs over a bucket held in registers by one team
        const size_t teams = (qc::kBlock / 32) / p.team_warps;
        if (!encode_tiles_for(p, esize, p.err != nullptr, grad16, tiles,
                              teams * qc::sel_region_words(p.bucket) * 4))
            return fail(QC_ERR_UNSUPPORTED,
                        "%s: percentile clipping needs a bucket of at most 4096 elements "
                        "and a 16-byte aligned gradient", fn);
        return from_cuda(qc::launch_encode_clip(p, tiles, bits, sr, bf16, st), fn);
    }
    if (bf16 && qc::encode_bf16_fast_applies(p, scheme, bits, sr, grad16, aligned(p.codes, 8)))
        return from_cuda(qc::launch_encode_bf16_fast(p, scheme, st), fn);
    // the bf16 kernel stores 8-bit codes eight bytes at a time
    if (bf16 && (bits != 8 || aligned(p.codes, 8)) && bf16_tiles_for(p, grad16, tiles))
        return from_cuda(qc::launch_encode_bf16(p, tiles, scheme, bits, sr, st), fn);
    if (encode_tiles_for(p, esize, p.err != nullptr, grad16, tiles))
        return from_cuda(qc::launch_encode_tma(p, tiles, scheme, bits, sr, bf16, st), fn);
    return from_cuda(qc::launch_encode(p, scheme, bits, sr, bf16, st), fn);
}

}  // namespace

extern "C" {

qc_status qc_encode_ef(const void *grad, qc_dtype dtype, float *err, size_t n, int bits,
                       size_t bucket, qc_scheme scheme, qc_round mode, uint64_t seed,
                       uint32_t step, uint32_t *codes, float *scale, float *offset,
                       qc_stream_t stream) {
    static const char *fn = "qc_encode_ef";
    qc_status sc = check_encode_args(fn, dtype, bits, bucket, scheme, mode);
    if (sc != QC_OK) return sc;
    if (n == 0) return ok();
    sc = check_encode_buffers(fn, grad, dtype, err, n, bits, bucket, scheme, codes, scale, offset);
    if (sc != QC_OK) return sc;
    qc::EncodeParams p = encode_params(bucket, seed, step);
    p.grad = grad;
    p.err = err;
    p.n = n;
    p.nbuckets = qc_num_buckets(n, bucket);
    p.codes = codes;
    p.scale = scale;
    p.offset = offset;
    return encode_one(fn, p, dtype, bits, scheme, mode, reinterpret_cast<cudaStream_t>(stream));
}

qc_status qc_encode_ef_segments(const qc_segment *segs, int nseg, qc_dtype dtype, int bits,
                                size_t bucket, qc_scheme scheme, qc_round mode, uint64_t seed,
                                uint32_t step, qc_stream_t stream) {
    static const char *fn = "qc_encode_ef_segments";
    qc_status sc = check_encode_args(fn, dtype, bits, bucket, scheme, mode);
    if (sc != QC_OK) return sc;
    if (nseg < 0) return fail(QC_ERR_INVALID_ARG, "%s: nseg must be >= 0 (got %d)", fn, nseg);
    if (nseg == 0) return ok();
    if (!segs) return fail(QC_ERR_NULL, "%s: segs must be non-NULL", fn);
    const bool uni = scheme == QC_SCHEME_UNIFORM || scheme == QC_SCHEME_UNIFORM_CLIP;
    const size_t esize = dtype == QC_DTYPE_F32 ? 4 : 2;
    bool any_err = false, all_err = true;
    uint64_t total = 0;
    for (int a = 0; a < nseg; ++a) {
        const qc_segment &g = segs[a];
        if (g.n == 0) continue;
        any_err |= g.err != nullptr;
        all_err &= g.err != nullptr;
        sc = check_encode_buffers(fn, g.grad, dtype, g.err, g.n, bits, bucket, scheme, g.codes,
                                  g.scale, g.offset);
        if (sc != QC_OK) {
            char msg[sizeof g_last_error];  // the message is rewritten into g_last_error
            snprintf(msg, sizeof msg, "%s", g_last_error);
            return fail(sc, "%.480s (segment %d)", msg, a);
        }
        total += g.n;
        if (total > (static_cast<uint64_t>(1) << 40))
            return fail(QC_ERR_UNSUPPORTED, "%s: the segments hold more than 2^40 elements", fn);
    }
    if (any_err && !all_err)
        return fail(QC_ERR_INVALID_ARG, "%s: err must be given for every segment or for none", fn);
    // no output of one segment may overlap any buffer of another
    for (int a = 0; a < nseg; ++a) {
        const qc_segment &x = segs[a];
        if (x.n == 0) continue;
        const size_t nb = qc_num_buckets(x.n, bucket);
        const void *outs[4] = {x.codes, x.scale, uni ? x.offset : nullptr, x.err};
        const size_t osz[4] = {qc_code_words(x.n, bits) * 4, nb * 4, nb * 4, x.n * 4};
        for (int b = 0; b < nseg; ++b) {
            const qc_segment &y = segs[b];
            if (b == a || y.n == 0) continue;
            const size_t mb = qc_num_buckets(y.n, bucket);
            const void *bufs[5] = {y.grad, y.err, y.codes, y.scale, uni ? y.offset : nullptr};
            const size_t bsz[5] = {y.n * esize, y.n * 4, qc_code_words(y.n, bits) * 4, mb * 4, mb * 4};
            for (int i = 0; i < 4; ++i)
                for (int j = 0; j < 5; ++j)
                    if (overlaps(outs[i], osz[i], bufs[j], bsz[j]))
                        return fail(QC_ERR_INVALID_ARG,
                                    "%s: an output of segment %d overlaps a buffer of segment %d", fn, a, b);
        }
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const qc::EncodeParams base = encode_params(bucket, seed, step);
    const bool sr = mode == QC_ROUND_STOCHASTIC, bf16 = dtype == QC_DTYPE_BF16;
    // the segment's own parameters, with its draw index base
    std::vector<qc::EncodeParams> ps;
    ps.reserve(static_cast<size_t>(nseg));
    uint64_t base_index = 0;
    for (int a = 0; a < nseg; ++a) {
        const qc_segment &g = segs[a];
        if (g.n == 0) continue;
        qc::EncodeParams p = base;
        p.grad = g.grad;
        p.err = g.err;
        p.n = g.n;
        p.nbuckets = qc_num_buckets(g.n, bucket);
        p.codes = g.codes;
        p.scale = g.scale;
        p.offset = g.offset;
        p.index_base = base_index;
        base_index += (g.n + 3u) & ~static_cast<uint64_t>(3);  // each segment starts a Philox block
        ps.push_back(p);
    }
    // Which one-launch kernel takes every segment: the receiver's bf16 kernel, or
    // the pipelined encode; otherwise each segment takes its own launch.
    bool fast = bf16, tma = scheme != QC_SCHEME_UNIFORM_CLIP;
    qc::EncodeTiles tiles{};
    for (const auto &p : ps) {
        fast = fast && qc::encode_bf16_fast_applies(p, scheme, bits, sr, aligned(p.grad, 16),
                                                    aligned(p.codes, 8));
        qc::EncodeTiles t{};
        tma = tma && encode_tiles_for(p, esize, any_err, aligned(p.grad, 16), t);
        if (tma) tiles = t;
    }
    if (fast || tma) {
        for (size_t first = 0; first < ps.size(); first += qc::kMaxSegments) {
            const size_t cnt = std::min(ps.size() - first, static_cast<size_t>(qc::kMaxSegments));
            qc::EncodeSegs S;
            S.nseg = static_cast<uint32_t>(cnt);
            uint64_t tile0 = 0;
            for (size_t i = 0; i < cnt; ++i) {
                const qc::EncodeParams &p = ps[first + i];
                S.s[i] = qc::EncodeSeg{p.grad, p.err, p.n, p.codes, p.scale, p.offset, tile0, p.index_base};
                tile0 += fast ? qc::encode_bf16_fast_tiles(p.n) : (p.n + tiles.te - 1) / tiles.te;
            }
            cudaError_t e;
            if (fast) {
                e = qc::launch_encode_bf16_fast(base, scheme, st, &S);
            } else {
                qc::EncodeTiles g = tiles;
                g.ntiles = tile0;
                qc::EncodeParams p = base;
                p.err = any_err ? ps[first].err : nullptr;  // selects the error-feedback kernel
                e = qc::launch_encode_tma(p, g, scheme, bits, sr, bf16, st, &S);
            }
            if (e != cudaSuccess) return from_cuda(e, fn);
        }
        return ok();
    }
    for (const auto &p : ps) {
        sc = encode_one(fn, p, dtype, bits, scheme, mode, st);
        if (sc != QC_OK) return sc;
    }
    return ok();
}

qc_status qc_decode_accumulate(const uint32_t *codes, size_t codes_stride_words,
                               const float *scale, const float *offset, size_t meta_stride,
                               int M, size_t n, int bits, size_t bucket, qc_scheme scheme,
                               float *out, int flags, qc_stream_t stream) {
    const qc_status sc = check_scheme("qc_decode_accumulate", scheme, bits);
    if (sc != QC_OK) return sc;
    // a percentile-clipped payload is a uniform payload over its clipped range
    if (scheme == QC_SCHEME_UNIFORM_CLIP) scheme = QC_SCHEME_UNIFORM;
    if (M < 1 || M > QC_MAX_WORKERS)
        return fail(QC_ERR_INVALID_ARG, "qc_decode_accumulate: M must be in [1, %d] (got %d)", QC_MAX_WORKERS, M);
    if (flags & ~(QC_OUT_MEAN | QC_ACCUMULATE_INTO_OUT))
        return fail(QC_ERR_INVALID_ARG, "qc_decode_accumulate: unknown flag bits 0x%x", flags);
    if (!valid_bucket(bucket))
        return fail(QC_ERR_INVALID_ARG, "qc_decode_accumulate: bucket must be a multiple of 32 in [32, 2^24] (got %zu)", bucket);
    if (n == 0) return ok();
    if (n > (static_cast<size_t>(1) << 40))
        return fail(QC_ERR_UNSUPPORTED, "qc_decode_accumulate: n = %zu exceeds 2^40 elements", n);
    const size_t words = qc_code_words(n, bits), nb = qc_num_buckets(n, bucket);
    if (M > 1 && (codes_stride_words < words || meta_stride < nb))
        return fail(QC_ERR_INVALID_ARG, "qc_decode_accumulate: strides (%zu words, %zu buckets) are shorter than one payload (%zu, %zu)",
                    codes_stride_words, meta_stride, words, nb);
    if (!codes || !scale || !out) return fail(QC_ERR_NULL, "qc_decode_accumulate: codes, scale and out must be non-NULL");
    if (scheme == QC_SCHEME_UNIFORM && !offset)
        return fail(QC_ERR_NULL, "qc_decode_accumulate: the uniform scheme needs offsets");
    if (!aligned(out, 16)) return fail(QC_ERR_ALIGNMENT, "qc_decode_accumulate: out must be 16-byte aligned");
    if (!aligned(codes, 4) || !aligned(scale, 4) || (offset && !aligned(offset, 4)))
        return fail(QC_ERR_ALIGNMENT, "qc_decode_accumulate: codes, scale and offset must be 4-byte aligned");
    const size_t span_c = ((M - 1) * (M > 1 ? codes_stride_words : 0) + words) * 4;
    const size_t span_m = ((M - 1) * (M > 1 ? meta_stride : 0) + nb) * 4;
    if (overlaps(out, n * 4, codes, span_c) || overlaps(out, n * 4, scale, span_m) ||
        (scheme == QC_SCHEME_UNIFORM && overlaps(out, n * 4, offset, span_m)))
        return fail(QC_ERR_INVALID_ARG, "qc_decode_accumulate: out overlaps an input");

    qc::DecodeParams p{};
    p.codes = codes;
    p.codes_stride = M > 1 ? codes_stride_words : 0;
    p.scale = scale;
    p.offset = offset;
    p.meta_stride = M > 1 ? meta_stride : 0;
    p.M = M;
    p.n = n;
    p.bucket = static_cast<uint32_t>(bucket);
    p.nbuckets = nb;
    p.out = out;
    p.flags = flags;
    // x / M and x * (1 / M) round the same exact value when M is a power of two.
    p.inv_m = (M & (M - 1)) == 0 ? 1.0f / static_cast<float>(M) : 0.0f;
    p.status = g_status_word;
    qc::DecodeTiles tiles{};
    if (decode_tiles_for(p, bits, tiles))
        return from_cuda(qc::launch_decode_tma(p, tiles, scheme, bits, reinterpret_cast<cudaStream_t>(stream)),
                         "qc_decode_accumulate");
    return from_cuda(qc::launch_decode(p, scheme, bits, reinterpret_cast<cudaStream_t>(stream)),
                     "qc_decode_accumulate");
}

qc_status qc_reencode(const uint32_t *codes, size_t codes_stride_words, const float *scale,
                      const float *offset, size_t meta_stride, int M, size_t n, int bits,
                      size_t bucket, qc_scheme scheme, int flags, float *err, qc_round mode,
                      uint64_t seed, uint32_t step, uint32_t *codes_out, float *scale_out,
                      float *offset_out, float *out, qc_stream_t stream) {
    static const char *fn = "qc_reencode";
    const qc_status sc = check_scheme(fn, scheme, bits);
    if (sc != QC_OK) return sc;
    if (scheme == QC_SCHEME_UNIFORM_CLIP)
        return fail(QC_ERR_UNSUPPORTED, "%s: percentile clipping is not fused into the re-encode; "
                    "use qc_decode_accumulate followed by qc_encode_ef", fn);
    if (mode != QC_ROUND_NEAREST && mode != QC_ROUND_STOCHASTIC)
        return fail(QC_ERR_INVALID_ARG, "%s: unknown rounding mode %d", fn, mode);
    if (scheme == QC_SCHEME_SIGN && mode != QC_ROUND_NEAREST)
        return fail(QC_ERR_INVALID_ARG, "%s: sign scheme is deterministic; mode must be NEAREST", fn);
    if (M < 1 || M > QC_MAX_WORKERS)
        return fail(QC_ERR_INVALID_ARG, "%s: M must be in [1, %d] (got %d)", fn, QC_MAX_WORKERS, M);
    if (flags & ~QC_OUT_MEAN)
        return fail(QC_ERR_INVALID_ARG, "%s: flags may hold only QC_OUT_MEAN (got 0x%x)", fn, flags);
    if (!valid_bucket(bucket))
        return fail(QC_ERR_INVALID_ARG, "%s: bucket must be a multiple of 32 in [32, 2^24] (got %zu)", fn, bucket);
    if (n == 0) return ok();
    if (n > (static_cast<size_t>(1) << 40))
        return fail(QC_ERR_UNSUPPORTED, "%s: n = %zu exceeds 2^40 elements", fn, n);
    const size_t words = qc_code_words(n, bits), nb = qc_num_buckets(n, bucket);
    if (M > 1 && (codes_stride_words < words || meta_stride < nb))
        return fail(QC_ERR_INVALID_ARG, "%s: strides (%zu words, %zu buckets) are shorter than one payload (%zu, %zu)",
                    fn, codes_stride_words, meta_stride, words, nb);
    if (!codes || !scale || !codes_out || !scale_out)
        return fail(QC_ERR_NULL, "%s: codes, scale, codes_out and scale_out must be non-NULL", fn);
    const bool uni = scheme == QC_SCHEME_UNIFORM;
    if (uni && (!offset || !offset_out))
        return fail(QC_ERR_NULL, "%s: the uniform scheme needs offset and offset_out", fn);
    if ((err && !aligned(err, 16)) || (out && !aligned(out, 16)))
        return fail(QC_ERR_ALIGNMENT, "%s: err and out must be 16-byte aligned", fn);
    if (!aligned(codes, 4) || !aligned(scale, 4) || (offset && !aligned(offset, 4)) ||
        !aligned(codes_out, 4) || !aligned(scale_out, 4) || (offset_out && !aligned(offset_out, 4)))
        return fail(QC_ERR_ALIGNMENT, "%s: code words and metadata must be 4-byte aligned", fn);
    const size_t span_c = ((M - 1) * (M > 1 ? codes_stride_words : 0) + words) * 4;
    const size_t span_m = ((M - 1) * (M > 1 ? meta_stride : 0) + nb) * 4;
    const void *ins[3] = {codes, scale, uni ? offset : nullptr};
    const size_t isz[3] = {span_c, span_m, span_m};
    const void *outs[5] = {codes_out, scale_out, uni ? offset_out : nullptr, err, out};
    const size_t osz[5] = {words * 4, nb * 4, nb * 4, n * 4, n * 4};
    for (int a = 0; a < 5; ++a) {
        for (int b = 0; b < 3; ++b)
            if (overlaps(outs[a], osz[a], ins[b], isz[b]))
                return fail(QC_ERR_INVALID_ARG, "%s: an output overlaps an input payload", fn);
        for (int b = a + 1; b < 5; ++b)
            if (overlaps(outs[a], osz[a], outs[b], osz[b]))
                return fail(QC_ERR_INVALID_ARG, "%s: outputs overlap each other", fn);
    }

    qc::ReencodeParams p{};
    p.codes = codes;
    p.codes_stride = M > 1 ? codes_stride_words : 0;
    p.scale = scale;
    p.offset = offset;
    p.meta_stride = M > 1 ? meta_stride : 0;
    p.M = M;
    p.n = n;
    p.bucket = static_cast<uint32_t>(bucket);
    p.nbuckets = nb;
    p.flags = flags;
    p.inv_m = (M & (M - 1)) == 0 ? 1.0f / static_cast<float>(M) : 0.0f;
    p.out = out;
    p.err = err;
    p.step = step;
    p.team_warps = team_warps_for(bucket);
    p.keys = qc::philox_round_keys(seed);
    p.codes_out = codes_out;
    p.scale_out = scale_out;
    p.offset_out = offset_out;
    p.status = g_status_word;
    qc::ReencodeTiles tiles{};
    if (!reencode_tiles_for(p, bits, tiles))
        return fail(QC_ERR_UNSUPPORTED,
                    "%s: needs 16-byte aligned codes, a worker stride that is a multiple of 4 words "
                    "and a bucket whose tile (a multiple of 128 elements) is at most 8192; "
                    "qc_decode_accumulate followed by qc_encode_ef computes the same result", fn);
    return from_cuda(qc::launch_reencode(p, tiles, scheme, bits, mode == QC_ROUND_STOCHASTIC,
                                         reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

qc_status qc_topk_encode_ef(const void *grad, qc_dtype dtype, float *err, size_t n, size_t bucket,
                            uint32_t keep, qc_round mode, uint64_t seed, uint32_t step,
                            uint32_t *idx, uint8_t *codes, float *scale, float *offset,
                            qc_stream_t stream) {
    static const char *fn = "qc_topk_encode_ef";
    if (dtype != QC_DTYPE_F32 && dtype != QC_DTYPE_BF16)
        return fail(QC_ERR_INVALID_ARG, "%s: dtype %d is not F32 or BF16", fn, dtype);
    if (mode != QC_ROUND_NEAREST && mode != QC_ROUND_STOCHASTIC)
        return fail(QC_ERR_INVALID_ARG, "%s: unknown rounding mode %d", fn, mode);
    if (!valid_bucket(bucket))
        return fail(QC_ERR_INVALID_ARG, "%s: bucket must be a multiple of 32 in [32, 2^24] (got %zu)", fn, bucket);
    if (keep < 1 || keep > bucket)
        return fail(QC_ERR_INVALID_ARG, "%s: keep must be in [1, bucket] (got %u)", fn, keep);
    if (bucket > 4096)
        return fail(QC_ERR_UNSUPPORTED, "%s: buckets above 4096 elements are not supported", fn);
    if (n == 0) return ok();
    if (n >= (static_cast<size_t>(1) << 32))
        return fail(QC_ERR_UNSUPPORTED, "%s: indices are 32-bit; n = %zu is too large", fn, n);
    if (!grad || !idx || !codes || !scale || !offset)
        return fail(QC_ERR_NULL, "%s: grad, idx, codes, scale and offset must be non-NULL", fn);
    const size_t esize = dtype == QC_DTYPE_F32 ? 4 : 2;
    if (!aligned(grad, 16))
        return fail(QC_ERR_UNSUPPORTED, "%s: the gradient must be 16-byte aligned", fn);
    if (err && !aligned(err, 16)) return fail(QC_ERR_ALIGNMENT, "%s: err must be 16-byte aligned", fn);
    if (!aligned(idx, 4) || !aligned(scale, 4) || !aligned(offset, 4))
        return fail(QC_ERR_ALIGNMENT, "%s: idx, scale and offset must be 4-byte aligned", fn);
    const size_t nb = qc_num_buckets(n, bucket), slots = nb * keep;
    const void *outs[4] = {idx, codes, scale, offset};
    const size_t osz[4] = {slots * 4, slots, nb * 4, nb * 4};
    for (int x = 0; x < 4; ++x) {
        if (overlaps(outs[x], osz[x], grad, n * esize) || overlaps(outs[x], osz[x], err, n * 4))
            return fail(QC_ERR_INVALID_ARG, "%s: an output overlaps grad or err", fn);
        for (int y = x + 1; y < 4; ++y)
            if (overlaps(outs[x], osz[x], outs[y], osz[y]))
                return fail(QC_ERR_INVALID_ARG, "%s: outputs overlap each other", fn);
    }
    if (overlaps(err, n * 4, grad, n * esize)) return fail(QC_ERR_INVALID_ARG, "%s: err overlaps grad", fn);

    qc::TopkParams t{};
    t.e.grad = grad;
    t.e.err = err;
    t.e.n = n;
    t.e.bucket = static_cast<uint32_t>(bucket);
    t.e.nbuckets = nb;
    t.e.team_warps = team_warps_for(bucket);
    t.e.two_pass = 0;
    t.e.seed = seed;
    t.e.step = step;
    t.e.keys = qc::philox_round_keys(seed);
    t.e.scale = scale;
    t.e.offset = offset;
    t.e.status = g_status_word;
    t.keep = keep;
    t.idx = idx;
    t.codes8 = codes;
    qc::EncodeTiles tiles{};
    const size_t teams = (qc::kBlock / 32) / t.e.team_warps;
    if (!encode_tiles_for(t.e, esize, err != nullptr, true, tiles,
                          teams * (qc::sel_region_words(t.e.bucket) + qc::kTopkScanWords) * 4))
        return fail(QC_ERR_UNSUPPORTED, "%s: no tiling for this bucket", fn);
    return from_cuda(qc::launch_topk_encode(t, tiles, mode == QC_ROUND_STOCHASTIC,
                                            dtype == QC_DTYPE_BF16,
                                            reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

qc_status qc_topk_decode_accumulate(const uint32_t *idx, const uint8_t *codes, size_t pair_stride,
                                    const float *scale, const float *offset, size_t meta_stride,
                                    int M, size_t n, size_t bucket, uint32_t keep, float *out,
                                    int flags, qc_stream_t stream) {
    static const char *fn = "qc_topk_decode_accumulate";
    if (M < 1 || M > QC_MAX_WORKERS)
        return fail(QC_ERR_INVALID_ARG, "%s: M must be in [1, %d] (got %d)", fn, QC_MAX_WORKERS, M);
    if (flags & ~(QC_OUT_MEAN | QC_ACCUMULATE_INTO_OUT))
        return fail(QC_ERR_INVALID_ARG, "%s: unknown flag bits 0x%x", fn, flags);
    if (!valid_bucket(bucket))
        return fail(QC_ERR_INVALID_ARG, "%s: bucket must be a multiple of 32 in [32, 2^24] (got %zu)", fn, bucket);
    if (keep < 1 || keep > bucket)
        return fail(QC_ERR_INVALID_ARG, "%s: keep must be in [1, bucket] (got %u)", fn, keep);
    if (bucket > 16384 || keep > 1024)
        return fail(QC_ERR_UNSUPPORTED, "%s: buckets above 16384 elements or keep above 1024 are not supported", fn);
    if (n == 0) return ok();
    if (n >= (static_cast<size_t>(1) << 32))
        return fail(QC_ERR_UNSUPPORTED, "%s: indices are 32-bit; n = %zu is too large", fn, n);
    const size_t nb = qc_num_buckets(n, bucket), slots = nb * keep;
    if (M > 1 && (pair_stride < slots || meta_stride < nb))
        return fail(QC_ERR_INVALID_ARG, "%s: strides (%zu slots, %zu buckets) are shorter than one payload (%zu, %zu)",
                    fn, pair_stride, meta_stride, slots, nb);
    if (!idx || !codes || !scale || !offset || !out)
        return fail(QC_ERR_NULL, "%s: idx, codes, scale, offset and out must be non-NULL", fn);
    if (!aligned(idx, 4) || !aligned(scale, 4) || !aligned(offset, 4) || !aligned(out, 4))
        return fail(QC_ERR_ALIGNMENT, "%s: idx, scale, offset and out must be 4-byte aligned", fn);
    const size_t ps = M > 1 ? pair_stride : 0, ms = M > 1 ? meta_stride : 0;
    const size_t span_p = (M - 1) * ps + slots, span_m = ((M - 1) * ms + nb) * 4;
    if (overlaps(out, n * 4, idx, span_p * 4) || overlaps(out, n * 4, codes, span_p) ||
        overlaps(out, n * 4, scale, span_m) || overlaps(out, n * 4, offset, span_m))
        return fail(QC_ERR_INVALID_ARG, "%s: out overlaps an input", fn);
    qc::TopkDecodeParams d{};
    d.idx = idx;
    d.codes8 = codes;
    d.pair_stride = ps;
    d.scale = scale;
    d.offset = offset;
    d.meta_stride = ms;
    d.M = M;
    d.n = n;
    d.bucket = static_cast<uint32_t>(bucket);
    d.nbuckets = nb;
    d.keep = keep;
    d.out = out;
    d.flags = flags;
    d.inv_m = (M & (M - 1)) == 0 ? 1.0f / static_cast<float>(M) : 0.0f;
    return from_cuda(qc::launch_topk_decode(d, reinterpret_cast<cudaStream_t>(stream)), fn);
}

qc_status qc_sign_vote(const uint32_t *signs, size_t stride_words, int M, size_t n,
                       uint32_t *out, qc_stream_t stream) {
    if (M < 1 || M > QC_MAX_WORKERS)
        return fail(QC_ERR_INVALID_ARG, "qc_sign_vote: M must be in [1, %d] (got %d)", QC_MAX_WORKERS, M);
    if (n == 0) return ok();
    if (n > (static_cast<size_t>(1) << 40))
        return fail(QC_ERR_UNSUPPORTED, "qc_sign_vote: n = %zu exceeds 2^40 elements", n);
    const size_t words = qc_code_words(n, 1);
    if (M > 1 && stride_words < words)
        return fail(QC_ERR_INVALID_ARG, "qc_sign_vote: stride %zu words is shorter than one vector (%zu)", stride_words, words);
    if (!signs || !out) return fail(QC_ERR_NULL, "qc_sign_vote: signs and out must be non-NULL");
    if (!aligned(signs, 4) || !aligned(out, 4))
        return fail(QC_ERR_ALIGNMENT, "qc_sign_vote: signs and out must be 4-byte aligned");
    const size_t stride = M > 1 ? stride_words : 0;
    if (overlaps(out, words * 4, signs, ((M - 1) * stride + words) * 4))
        return fail(QC_ERR_INVALID_ARG, "qc_sign_vote: out overlaps the inputs");
    qc::VoteParams p{};
    p.signs = signs;
    p.stride = stride;
    p.M = M;
    p.nwords = words;
    p.threshold = static_cast<uint32_t>((M + 1) / 2);
    p.last_mask = (n % 32) ? ((1u << (n % 32)) - 1u) : 0xFFFFFFFFu;
    p.out = out;
    const bool vec = aligned(signs, 16) && aligned(out, 16) && stride % 4 == 0;
    return from_cuda(qc::launch_vote(p, vec, reinterpret_cast<cudaStream_t>(stream)), "qc_sign_vote");
}

static qc_status check_fp8(const char *fn, const void *in, const void *codes, const float *sc,
                           size_t rows, size_t dim, const void *out_f32) {
    if (dim < 4 || dim % 4 != 0)
        return fail(QC_ERR_INVALID_ARG, "%s: dim must be a positive multiple of 4 (got %zu)", fn, dim);
    if (dim > QC_MAX_FP8_DIM)
        return fail(QC_ERR_UNSUPPORTED, "%s: dim %zu exceeds %d", fn, dim, QC_MAX_FP8_DIM);
    if (rows == 0) return QC_OK;
    if (rows > (static_cast<size_t>(1) << 40) / dim)
        return fail(QC_ERR_UNSUPPORTED, "%s: rows x dim exceeds 2^40", fn);
    if (!in || !codes || !sc) return fail(QC_ERR_NULL, "%s: a buffer pointer is NULL", fn);
    if (!aligned(out_f32, 16)) return fail(QC_ERR_ALIGNMENT, "%s: the fp32 buffer must be 16-byte aligned", fn);
    if (!aligned(codes, 4) || !aligned(sc, 4))
        return fail(QC_ERR_ALIGNMENT, "%s: codes and row_scale must be 4-byte aligned", fn);
    return QC_OK;
}

qc_status qc_rowwise_fp8(const float *x, size_t rows, size_t dim, uint8_t *codes,
                         float *row_scale, qc_stream_t stream) {
    qc_status st = check_fp8("qc_rowwise_fp8", x, codes, row_scale, rows, dim, x);
    if (st != QC_OK) return st;
    if (rows == 0) return ok();
    if (overlaps(codes, rows * dim, x, rows * dim * 4) || overlaps(row_scale, rows * 4, x, rows * dim * 4) ||
        overlaps(codes, rows * dim, row_scale, rows * 4))
        return fail(QC_ERR_INVALID_ARG, "qc_rowwise_fp8: buffers overlap");
    qc::Fp8Params p{};
    p.x = x;
    p.rows = rows;
    p.dim = static_cast<uint32_t>(dim);
    p.team_warps = team_warps_for(dim);
    p.codes = codes;
    p.row_scale = row_scale;
    return from_cuda(qc::launch_fp8_quant(p, reinterpret_cast<cudaStream_t>(stream)), "qc_rowwise_fp8");
}

qc_status qc_rowwise_fp8_dequant(const uint8_t *codes, const float *row_scale, size_t rows,
                                 size_t dim, float *out, qc_stream_t stream) {
    qc_status st = check_fp8("qc_rowwise_fp8_dequant", out, codes, row_scale, rows, dim, out);
    if (st != QC_OK) return st;
    if (rows == 0) return ok();
    if (overlaps(out, rows * dim * 4, codes, rows * dim) || overlaps(out, rows * dim * 4, row_scale, rows * 4))
        return fail(QC_ERR_INVALID_ARG, "qc_rowwise_fp8_dequant: out overlaps an input");
    qc::Fp8Params p{};
    p.codes_in = codes;
    p.scale_in = row_scale;
    p.rows = rows;
    p.dim = static_cast<uint32_t>(dim);
    p.team_warps = team_warps_for(dim);
    p.out = out;
    return from_cuda(qc::launch_fp8_dequant(p, reinterpret_cast<cudaStream_t>(stream)),
                     "qc_rowwise_fp8_dequant");
}

}  // extern "C"
