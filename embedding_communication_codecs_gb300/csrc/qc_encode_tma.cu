// qc_encode_tma.cu -- instances of the pipelined encode kernel (the kernel
// template lives in qc_encode_tma.cuh) for the uniform, sign, ternary and QSGD
// schemes.
//
// "Quantization for Communication", "Quantization Schemes", "Quantized SGD
// Algorithms", "Error Feedback for Quantization", "Hardware Acceleration" (the
// arithmetic is the shared code in qc_encode_math.cuh).
//
// A tile is TB whole buckets (TE = TB * bucket elements, about 24-32 KB of
// input).  Each persistent block owns tiles blockIdx.x, blockIdx.x + grid, ...;
// thread 0 keeps `stages - 1` tiles of copies in flight ahead of the one being
// quantized, so the bytes in flight per SM no longer depend on registers.  The
// compute side is the team layout of the direct kernel, reading its slots from
// shared memory; codes, residuals and metadata are stored straight from
// registers.  Tail bytes that are not a whole 16-byte unit (n % 4 != 0 for
// fp32) are read from global memory directly.
#include "qc_encode_tma.cuh"

namespace qc {

cudaError_t launch_encode_tma(const EncodeParams &p, const EncodeTiles &g, int scheme, int bits,
                              int stochastic, int bf16, cudaStream_t stream,
                              const EncodeSegs *segs) {
    if (scheme == kLog) return launch_encode_log(p, g, bits, stochastic, bf16, stream, segs);
    if (scheme == kSign) return launch_dtype<kSign, 1, false>(p, g, bf16, stream, segs);
    if (scheme == kTernary) return launch_round<kTernary, 2>(p, g, stochastic, bf16, stream, segs);
    if (scheme == kQsgd) {
        if (bits == 2) return launch_round<kQsgd, 2>(p, g, stochastic, bf16, stream, segs);
        if (bits == 4) return launch_round<kQsgd, 4>(p, g, stochastic, bf16, stream, segs);
        return launch_round<kQsgd, 8>(p, g, stochastic, bf16, stream, segs);
    }
    switch (bits) {
        case 1: return launch_round<kUniform, 1>(p, g, stochastic, bf16, stream, segs);
        case 2: return launch_round<kUniform, 2>(p, g, stochastic, bf16, stream, segs);
        case 4: return launch_round<kUniform, 4>(p, g, stochastic, bf16, stream, segs);
        default: return launch_round<kUniform, 8>(p, g, stochastic, bf16, stream, segs);
    }
}

QC_DEFINE_TAKE_FLAG(take_encode_errors, g_encode_errors)

}  // namespace qc
