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
// instantiations of the common kernel file compiling in parallel; the bf16
// instances live in qc_encode_clip_bf16.cu.
#include "qc_encode_tma.cuh"

namespace qc {

namespace {

template <int BITS, bool SR>
cudaError_t launch_f32(const EncodeParams &p, const EncodeTiles &g, cudaStream_t stream) {
    return p.err ? launch_one<kClip, BITS, SR, float, true>(p, g, stream, nullptr)
                 : launch_one<kClip, BITS, SR, float, false>(p, g, stream, nullptr);
}

template <int BITS>
cudaError_t launch_bits(const EncodeParams &p, const EncodeTiles &g, int stochastic,
                        cudaStream_t stream) {
    return stochastic ? launch_f32<BITS, true>(p, g, stream) : launch_f32<BITS, false>(p, g, stream);
}

}  // namespace

// fp32 gradients here; bf16 gradients in qc_encode_clip_bf16.cu (the two halves
// compile in parallel)
cudaError_t launch_encode_clip(const EncodeParams &p, const EncodeTiles &g, int bits,
                               int stochastic, int bf16, cudaStream_t stream) {
    if (bf16) return launch_encode_clip_bf16(p, g, bits, stochastic, stream);
    switch (bits) {
        case 1: return launch_bits<1>(p, g, stochastic, stream);
        case 2: return launch_bits<2>(p, g, stochastic, stream);
        case 4: return launch_bits<4>(p, g, stochastic, stream);
        default: return launch_bits<8>(p, g, stochastic, stream);
    }
}

QC_DEFINE_TAKE_FLAG(take_encode_clip_errors, g_encode_errors)

}  // namespace qc
