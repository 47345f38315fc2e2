// qc_encode.cu -- instances of the direct encode kernel (qc_encode_direct.cuh)
// for the uniform, sign, ternary and QSGD schemes; the logarithmic levels are
// instantiated in qc_encode_direct_log.cu (the two compile in parallel).  The
// direct kernel serves buckets larger than the pipelined kernels' team window
// (two passes, the second read hitting L2) and gradients whose base is not
// 16-byte aligned.
#include "qc_encode_direct.cuh"

namespace qc {

// The logarithmic-level instances (qc_encode_direct_log.cu).
cudaError_t launch_encode_direct_log(const EncodeParams &p, int bits, int stochastic, int bf16,
                                     cudaStream_t stream);

cudaError_t launch_encode(const EncodeParams &p, int scheme, int bits, int stochastic, int bf16,
                          cudaStream_t stream) {
    if (scheme == kLog) return launch_encode_direct_log(p, bits, stochastic, bf16, stream);
    if (scheme == kSign) return launch_dtype<kSign, 1, false>(p, bf16, stream);
    if (scheme == kTernary) return launch_round<kTernary, 2>(p, stochastic, bf16, stream);
    if (scheme == kQsgd) {
        if (bits == 2) return launch_round<kQsgd, 2>(p, stochastic, bf16, stream);
        if (bits == 4) return launch_round<kQsgd, 4>(p, stochastic, bf16, stream);
        return launch_round<kQsgd, 8>(p, stochastic, bf16, stream);
    }
    switch (bits) {
        case 1: return launch_round<kUniform, 1>(p, stochastic, bf16, stream);
        case 2: return launch_round<kUniform, 2>(p, stochastic, bf16, stream);
        case 4: return launch_round<kUniform, 4>(p, stochastic, bf16, stream);
        default: return launch_round<kUniform, 8>(p, stochastic, bf16, stream);
    }
}

}  // namespace qc
