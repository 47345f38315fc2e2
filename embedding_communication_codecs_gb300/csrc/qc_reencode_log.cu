// qc_reencode_log.cu -- the logarithmic-level instances of the fused receiver
// re-encode (qc_reencode.cu has the method's description; the level rule is
// quantize<kLog> in qc_encode_math.cuh, "Quantization Schemes", Non-Uniform
// Quantization).
#include "qc_reencode.cuh"

namespace qc {

cudaError_t launch_reencode_log(const ReencodeParams &p, const ReencodeTiles &g, int bits,
                                int stochastic, cudaStream_t stream) {
    if (bits == 2) return launch_round<kLog, 2>(p, g, stochastic, stream);
    if (bits == 4) return launch_round<kLog, 4>(p, g, stochastic, stream);
    return launch_round<kLog, 8>(p, g, stochastic, stream);
}

QC_DEFINE_TAKE_FLAG(take_reencode_log_errors, g_reencode_errors)

}  // namespace qc
