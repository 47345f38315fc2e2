// qc_reencode.cu -- receiver re-encode: the owner of a shard decodes the M
// workers' payloads of that shard, accumulates them in the fixed worker order,
// and quantizes the result again, with its own error-feedback residual, for the
// second (all-gather) phase of a two-phase quantized all-reduce.
//
// "Quantization for Communication", "Quantization-Aware All-Reduce" (dequantize
// after the exchange, accumulate in higher precision, quantize for the next
// hop) and "Gradient Compression and Quantised Collectives" (the reduce-scatter
// and all-gather halves of the ring).  Per element:
//   r = sum over w = 0 .. M-1 of d_w (fixed order, fp32), optionally fl(r / M)
//   p = err ? fl(err + r) : r, then the encoder's per-bucket statistics,
//   quantization and residual with the same scheme, bits and bucket.
//
// One kernel, warp-specialised like the pipelined decode: warp 8 streams the
// code words (TMA bulk copies) and the per-bucket metadata (4-byte cp.async)
// into the stages; warps 0-7 consume.  A tile is TB whole buckets (TE
// elements, 4096 where the bucket allows); its workers arrive in chunks of MC
// per stage, so any M streams through the same stages.  The running sums live
// in shared memory (two TE-element buffers, alternating between tiles), which
// keeps the exact worker order across chunks.  After a tile's last chunk the consumers meet on a named
// barrier (which also agrees that every wait succeeded) and encode the tile from
// the sum buffer with the team layout of the encode kernels.  Every wait is
// bounded and a timeout is recorded in a device flag.
#include "qc_reencode.cuh"

namespace qc {

// The uniform scheme here; sign, ternary and QSGD in qc_reencode_other.cu (the
// two halves compile in parallel).
cudaError_t launch_reencode(const ReencodeParams &p, const ReencodeTiles &g, int scheme, int bits,
                            int stochastic, cudaStream_t stream) {
    if (scheme != kUniform) return launch_reencode_other(p, g, scheme, bits, stochastic, stream);
    switch (bits) {
        case 1: return launch_round<kUniform, 1>(p, g, stochastic, stream);
        case 2: return launch_round<kUniform, 2>(p, g, stochastic, stream);
        case 4: return launch_round<kUniform, 4>(p, g, stochastic, stream);
        default: return launch_round<kUniform, 8>(p, g, stochastic, stream);
    }
}

QC_DEFINE_TAKE_FLAG(take_reencode_errors, g_reencode_errors)

}  // namespace qc
