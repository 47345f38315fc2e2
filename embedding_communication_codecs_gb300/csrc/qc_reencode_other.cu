// qc_reencode_other.cu -- the sign, ternary and QSGD instances of the fused
// receiver re-encode (qc_reencode.cu has the method's description and the
// uniform instances; both instantiate the kernel template of qc_reencode.cuh).
#include "qc_reencode.cuh"

namespace qc {

cudaError_t launch_reencode_other(const ReencodeParams &p, const ReencodeTiles &g, int scheme,
                                  int bits, int stochastic, cudaStream_t stream) {
    if (scheme == kLog) return launch_reencode_log(p, g, bits, stochastic, stream);
    if (scheme == kSign) return launch_ef<kSign, 1, false>(p, g, stream);
    if (scheme == kTernary) return launch_round<kTernary, 2>(p, g, stochastic, stream);
    if (bits == 2) return launch_round<kQsgd, 2>(p, g, stochastic, stream);
    if (bits == 4) return launch_round<kQsgd, 4>(p, g, stochastic, stream);
    return launch_round<kQsgd, 8>(p, g, stochastic, stream);
}

QC_DEFINE_TAKE_FLAG(take_reencode_other_errors, g_reencode_errors)

}  // namespace qc
