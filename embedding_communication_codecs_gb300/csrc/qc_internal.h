// qc_internal.h -- launchers behind the C ABI (host side, C++ linkage).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qc {

enum Scheme : int { kUniform = 0, kSign = 1, kTernary = 2, kQsgd = 3, kClip = 4, kLog = 5 };

// Elements a team of W warps covers per window: 4 float4 slots per lane.
constexpr int kSlots = 4;
constexpr int kBlock = 256;
constexpr int kWindowPerWarp = kSlots * 4 * 32;  // 512

// Round keys of Philox4x32-10 for one seed: round r uses (a[r], b[r]) =
// (seed low + r * 0x9E3779B9, seed high + r * 0xBB67AE85), mod 2^32.
struct PhiloxKeys {
    uint32_t a[10], b[10];
};

inline PhiloxKeys philox_round_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        k.a[r] = k0;
        k.b[r] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return k;
}

struct EncodeParams {
    const void *grad;
    float *err;
    uint64_t n;
    uint32_t bucket;
    uint64_t nbuckets;
    int team_warps;   // 1, 2, 4 or 8 warps own one bucket
    int two_pass;     // bucket > 512 * team_warps: statistics pass, then re-read
    uint64_t seed;
    uint32_t step;
    PhiloxKeys keys;  // round keys of `seed`
    uint32_t *codes;
    float *scale;
    float *offset;
    uint32_t *status;  // the caller's status word (qc_set_status_word), or null
    uint64_t index_base = 0;  // draw index of element 0 (a segment's place in its call)
};

// Several flat gradients encoded by one launch ("segments"): each with its own
// arrays and length, its buckets starting at its own element 0; tiles never
// straddle two segments, and segment s owns the launch's tiles [tile0, tile0 +
// its tile count).  Stochastic draws of element i of a segment use the index
// index_base + i (with the call's one seed; index_base is a multiple of 4, so a
// segment's groups of four draws are whole Philox blocks).  A single array is
// one segment at index 0.
// Passed by value as a kernel parameter (60 segments: about 3.4 KB).
constexpr int kMaxSegments = 60;  // QC_MAX_SEGMENTS_PER_LAUNCH

struct EncodeSeg {
    const void *grad;
    float *err;
    uint64_t n;
    uint32_t *codes;
    float *scale;
    float *offset;
    uint64_t tile0;
    uint64_t index_base;
};

struct EncodeSegs {
    uint32_t nseg;
    EncodeSeg s[kMaxSegments];
};

// The segment table of a single-array call.
inline EncodeSegs single_segment(const EncodeParams &p) {
    EncodeSegs t;
    t.nseg = 1;
    t.s[0] = EncodeSeg{p.grad, p.err, p.n, p.codes, p.scale, p.offset, 0, p.index_base};
    return t;
}

// Tiling of the TMA-pipelined encode: TB whole buckets per tile (TE elements),
// `stages` shared-memory stages of stage_bytes each; the residual's part of a
// stage starts at e_offset.
struct EncodeTiles {
    uint32_t warps;  // warps per bucket (the bf16 kernel's own team size)
    uint32_t tb;
    uint32_t te;
    uint32_t stages;
    uint32_t stage_bytes;
    uint32_t e_offset;
    uint64_t ntiles;
};

// Stages, then the full and empty barriers, then the team-reduction buffer.
inline size_t encode_tiles_smem(const EncodeTiles &g, size_t stats_bytes) {
    return static_cast<size_t>(g.stages) * g.stage_bytes + 16u * g.stages + 2u * 8u * stats_bytes;
}

// Warp-specialised blocks: 8 consumer warps and one producer warp.
constexpr int kConsumerWarps = 8;
constexpr int kProducerBlock = (kConsumerWarps + 1) * 32;

struct DecodeParams {
    const uint32_t *codes;
    uint64_t codes_stride;  // words
    const float *scale;
    const float *offset;
    uint64_t meta_stride;   // floats
    int M;
    uint64_t n;
    uint32_t bucket;
    uint64_t nbuckets;
    float *out;
    int flags;
    float inv_m;  // 1 / M when M is a power of two (an exact multiply), else 0
    uint32_t *status;  // the caller's status word, or null
};

// Tiling of the pipelined decode: TB whole buckets (TE elements) per tile; a
// stage holds M slices of worker_bytes code bytes, then M x TB scales and
// M x TB offsets at meta_offset.  bucket_shift = log2(bucket) when the bucket
// is a power of two, else -1.
struct DecodeTiles {
    uint32_t tb;
    uint32_t te;
    uint32_t stages;
    uint32_t stage_bytes;
    uint32_t worker_bytes;
    uint32_t meta_offset;
    int bucket_shift;
    uint64_t ntiles;
};

inline size_t decode_tiles_smem(const DecodeTiles &g) {
    return static_cast<size_t>(g.stages) * g.stage_bytes + 16u * g.stages;
}

struct VoteParams {
    const uint32_t *signs;
    uint64_t stride;        // words
    int M;
    uint64_t nwords;
    uint32_t threshold;     // ceil(M / 2)
    uint32_t last_mask;     // valid bits of the last word
    uint32_t *out;
};

// Shared-memory words of one team's order-statistic selection (percentile
// clipping, top-k): histogram sets, short lists, counters, results, then two
// candidate lists of bucket / 4 keys each (layout in qc_encode_math.cuh).
constexpr int kSelFixedWords = 908;
__host__ __device__ constexpr int sel_region_words(uint32_t bucket) {
    return kSelFixedWords + 2 * static_cast<int>(bucket / 4u);
}
// Words of one team's scan totals in the top-k kernel (one per slot and warp).
constexpr int kTopkScanWords = 4 * 8;

// Top-k sparsification: the encode parameters plus the kept count per bucket
// and the index / 8-bit code outputs (keep slots per bucket).
struct TopkParams {
    EncodeParams e;
    uint32_t keep;
    uint32_t *idx;
    uint8_t *codes8;
};

// Receiver of top-k payloads: M workers' (index, code) slots at pair_stride,
// metadata at meta_stride; a dense fp32 output.
struct TopkDecodeParams {
    const uint32_t *idx;
    const uint8_t *codes8;
    uint64_t pair_stride;
    const float *scale;
    const float *offset;
    uint64_t meta_stride;
    int M;
    uint64_t n;
    uint32_t bucket;
    uint64_t nbuckets;
    uint32_t keep;
    float *out;
    int flags;
    float inv_m;
};

// Receiver re-encode: the decode of M payloads (DecodeParams' fields) feeding an
// encode of the result with its own residual buffer, same scheme, bits and bucket.
struct ReencodeParams {
    const uint32_t *codes;
    uint64_t codes_stride;  // words
    const float *scale;
    const float *offset;
    uint64_t meta_stride;   // floats
    int M;
    uint64_t n;
    uint32_t bucket;
    uint64_t nbuckets;
    int flags;
    float inv_m;
    float *out;             // the decoded result r, or null
    float *err;             // the receiver's residual (in/out), or null
    uint32_t step;
    int team_warps;
    PhiloxKeys keys;
    uint32_t *codes_out;
    float *scale_out;
    float *offset_out;
    uint32_t *status;       // the caller's status word, or null
};

// Tiling of the re-encode: TB whole buckets (TE elements) per tile, the M
// workers in chunks of MC per stage (nchunks stages per tile).  A stage holds MC
// slices of worker_bytes code bytes, then MC x TB (scale, offset) pairs at
// meta_offset.  Two TE-element fp32 buffers hold the running sums.
struct ReencodeTiles {
    uint32_t tb;
    uint32_t te;
    uint32_t mc;
    uint32_t nchunks;
    uint32_t stages;
    uint32_t stage_bytes;
    uint32_t worker_bytes;
    uint32_t meta_offset;
    int bucket_shift;
    uint64_t ntiles;
};

// Stages, the two sum buffers, the full and empty barriers, the team-reduction buffer.
inline size_t reencode_tiles_smem(const ReencodeTiles &g, size_t stats_bytes) {
    return static_cast<size_t>(g.stages) * g.stage_bytes + 2u * 4u * g.te + 16u * g.stages +
           2u * 8u * stats_bytes;
}

struct Fp8Params {
    const float *x;
    const uint8_t *codes_in;
    uint64_t rows;
    uint32_t dim;
    int team_warps;         // warps per row when dim > 128
    uint8_t *codes;
    float *row_scale;
    const float *scale_in;
    float *out;
};

// Each launcher picks the template instance and a persistent grid, launches on
// `stream` and returns cudaGetLastError().
cudaError_t launch_encode(const EncodeParams &p, int scheme, int bits, int stochastic,
                          int bf16, cudaStream_t stream);
cudaError_t launch_encode_tma(const EncodeParams &p, const EncodeTiles &g, int scheme, int bits,
                              int stochastic, int bf16, cudaStream_t stream,
                              const EncodeSegs *segs = nullptr);
// The percentile-clipped uniform scheme (its own translation unit).
cudaError_t launch_encode_clip(const EncodeParams &p, const EncodeTiles &g, int bits,
                               int stochastic, int bf16, cudaStream_t stream);
cudaError_t launch_encode_clip_bf16(const EncodeParams &p, const EncodeTiles &g, int bits,
                                    int stochastic, cudaStream_t stream);
// The logarithmic-level scheme in the pipelined kernel (its own translation unit).
cudaError_t launch_encode_log(const EncodeParams &p, const EncodeTiles &g, int bits,
                              int stochastic, int bf16, cudaStream_t stream,
                              const EncodeSegs *segs = nullptr);
cudaError_t launch_encode_bf16(const EncodeParams &p, const EncodeTiles &g, int scheme, int bits,
                               int stochastic, cudaStream_t stream);
// The receiver's bf16 encodes without error feedback for buckets of 1024
// (8-bit nearest, ternary stochastic): whether they apply, and the launch.
bool encode_bf16_fast_applies(const EncodeParams &p, int scheme, int bits, int stochastic,
                              bool grad16, bool codes8);
cudaError_t launch_encode_bf16_fast(const EncodeParams &p, int scheme, cudaStream_t stream,
                                    const EncodeSegs *segs = nullptr);
// Tiles of the receiver kernel over n elements (a segment's share of a launch).
uint64_t encode_bf16_fast_tiles(uint64_t n);
cudaError_t launch_decode(const DecodeParams &p, int scheme, int bits, cudaStream_t stream);
cudaError_t launch_decode_tma(const DecodeParams &p, const DecodeTiles &g, int scheme, int bits,
                              cudaStream_t stream);
cudaError_t launch_reencode(const ReencodeParams &p, const ReencodeTiles &g, int scheme, int bits,
                            int stochastic, cudaStream_t stream);
cudaError_t launch_reencode_other(const ReencodeParams &p, const ReencodeTiles &g, int scheme,
                                  int bits, int stochastic, cudaStream_t stream);
cudaError_t launch_reencode_log(const ReencodeParams &p, const ReencodeTiles &g, int bits,
                                int stochastic, cudaStream_t stream);
cudaError_t launch_topk_encode(const TopkParams &p, const EncodeTiles &g, int stochastic, int bf16,
                               cudaStream_t stream);
cudaError_t launch_topk_decode(const TopkDecodeParams &p, cudaStream_t stream);
cudaError_t launch_vote(const VoteParams &p, bool vectorised, cudaStream_t stream);
cudaError_t launch_fp8_quant(const Fp8Params &p, cudaStream_t stream);
cudaError_t launch_fp8_dequant(const Fp8Params &p, cudaStream_t stream);

// Persistent grid: min(work units, SMs x resident blocks of `kernel` with
// `smem` bytes of dynamic shared memory).
int persistent_grid(const void *kernel, int block, uint64_t units, size_t smem = 0);

// Raises the kernel's dynamic shared memory limit to `bytes` (once per device).
cudaError_t prepare_dynamic_smem(const void *kernel, size_t bytes);

// Device-side error flags of the pipelined kernels: each stores its flag in
// *flags and clears it (one atomic exchange), returning the CUDA status.
cudaError_t take_encode_errors(uint32_t *flags);
cudaError_t take_encode_clip_errors(uint32_t *flags);
cudaError_t take_encode_clip_bf16_errors(uint32_t *flags);
cudaError_t take_encode_log_errors(uint32_t *flags);
cudaError_t take_reencode_other_errors(uint32_t *flags);
cudaError_t take_reencode_log_errors(uint32_t *flags);
cudaError_t take_selftest_errors(uint32_t *flags);

// One block waits on a barrier nothing completes for timeout_us microseconds,
// and records the pipeline-timeout flag (and *status, if given) (qc_selftest.cu).
cudaError_t launch_wait_timeout_selftest(uint32_t timeout_us, uint32_t *status, cudaStream_t stream);
cudaError_t take_topk_errors(uint32_t *flags);
cudaError_t take_encode_bf16_errors(uint32_t *flags);
cudaError_t take_encode_bf16_fast_errors(uint32_t *flags);
cudaError_t take_decode_errors(uint32_t *flags);
cudaError_t take_reencode_errors(uint32_t *flags);

}  // namespace qc
