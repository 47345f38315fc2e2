// qc_encode_log.cu -- instances of the pipelined encode kernel (qc_encode_tma.cuh)
// for the logarithmic-level scheme.
//
// "Quantization for Communication", "Quantization Schemes" (Non-Uniform
// Quantization: logarithmic levels, more levels near zero, dequantization
// through a lookup table).  A b-bit code is a sign bit over the index j of the
// level s * 2^(j - J) (J = 2^(b-1) - 1, level 0 is zero), s = max |p| of the
// bucket; the arithmetic is quantize<kLog> in qc_encode_math.cuh (exact: the
// division |p| / s, then the quotient's exponent and mantissa).
#include "qc_encode_tma.cuh"

namespace qc {

cudaError_t launch_encode_log(const EncodeParams &p, const EncodeTiles &g, int bits,
                              int stochastic, int bf16, cudaStream_t stream,
                              const EncodeSegs *segs) {
    if (bits == 2) return launch_round<kLog, 2>(p, g, stochastic, bf16, stream, segs);
    if (bits == 4) return launch_round<kLog, 4>(p, g, stochastic, bf16, stream, segs);
    return launch_round<kLog, 8>(p, g, stochastic, bf16, stream, segs);
}

QC_DEFINE_TAKE_FLAG(take_encode_log_errors, g_encode_errors)

}  // namespace qc
