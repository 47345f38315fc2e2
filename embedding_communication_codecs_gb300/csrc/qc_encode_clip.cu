// qc_encode_clip.cu -- instances of the pipelined encode kernel
// (qc_encode_tma.cuh) for uniform quantization over a percentile-clipped range.
//
// "Quantization for Communication", "Adaptive Quantization Strategies"
// (Percentile Clipping: set min and max to the 1st and 99th percentiles rather
// than the absolute extremes, so outliers do not waste the quantization range).
// Each team finds its bucket's two nearest-rank percentiles by radix selection
// over the slots it already holds in registers (team_percentiles in
// qc_encode_math.cuh), clamps every element into that range and quantizes it
// with the uniform scheme's arithmetic; with error feedback the residual
// p - deq keeps the clipped part.  A separate translation unit keeps the
// instantiations of the common kernel file compiling in parallel.
#include "qc_encode_tma.cuh"

namespace qc {

cudaError_t launch_encode_clip(const EncodeParams &p, const EncodeTiles &g, int bits,
                               int stochastic, int bf16, cudaStream_t stream) {
    switch (bits) {
        case 1: return launch_round<kClip, 1>(p, g, stochastic, bf16, stream);
        case 2: return launch_round<kClip, 2>(p, g, stochastic, bf16, stream);
        case 4: return launch_round<kClip, 4>(p, g, stochastic, bf16, stream);
        default: return launch_round<kClip, 8>(p, g, stochastic, bf16, stream);
    }
}

uint32_t take_encode_clip_errors() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_encode_errors, sizeof v);
    cudaMemcpyToSymbol(g_encode_errors, &zero, sizeof zero);
    return v;
}

}  // namespace qc
