// qc_encode_clip_bf16.cu -- the bf16-gradient instances of the percentile-
// clipped uniform encode (qc_encode_clip.cu has the method's description and the
// fp32 instances; both instantiate the kernel template of qc_encode_tma.cuh).
#include "qc_encode_tma.cuh"

namespace qc {

namespace {

template <int BITS, bool SR>
cudaError_t launch_b16(const EncodeParams &p, const EncodeTiles &g, cudaStream_t stream) {
    return p.err ? launch_one<kClip, BITS, SR, uint16_t, true>(p, g, stream, nullptr)
                 : launch_one<kClip, BITS, SR, uint16_t, false>(p, g, stream, nullptr);
}

template <int BITS>
cudaError_t launch_bits(const EncodeParams &p, const EncodeTiles &g, int stochastic,
                        cudaStream_t stream) {
    return stochastic ? launch_b16<BITS, true>(p, g, stream) : launch_b16<BITS, false>(p, g, stream);
}

}  // namespace

cudaError_t launch_encode_clip_bf16(const EncodeParams &p, const EncodeTiles &g, int bits,
                                    int stochastic, cudaStream_t stream) {
    switch (bits) {
        case 1: return launch_bits<1>(p, g, stochastic, stream);
        case 2: return launch_bits<2>(p, g, stochastic, stream);
        case 4: return launch_bits<4>(p, g, stochastic, stream);
        default: return launch_bits<8>(p, g, stochastic, stream);
    }
}

QC_DEFINE_TAKE_FLAG(take_encode_clip_bf16_errors, g_encode_errors)

}  // namespace qc
