// qc_encode_direct_log.cu -- instances of the direct encode kernel
// (qc_encode_direct.cuh) for the logarithmic-level scheme ("Quantization
// Schemes", Non-Uniform Quantization; the level rule is quantize<kLog> in
// qc_encode_math.cuh).
#include "qc_encode_direct.cuh"

namespace qc {

cudaError_t launch_encode_direct_log(const EncodeParams &p, int bits, int stochastic, int bf16,
                                     cudaStream_t stream) {
    if (bits == 2) return launch_round<kLog, 2>(p, stochastic, bf16, stream);
    if (bits == 4) return launch_round<kLog, 4>(p, stochastic, bf16, stream);
    return launch_round<kLog, 8>(p, stochastic, bf16, stream);
}

}  // namespace qc
