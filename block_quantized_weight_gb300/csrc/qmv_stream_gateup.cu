// qmv_stream_gateup.cu -- instantiations of the streaming M = 1 kernel for the fused Q4_0 gate+up (two matrices).
// Split into its own translation unit so the build compiles the variants in parallel.
#include "qmv_stream.cuh"

namespace qbw {

cudaError_t launch_stream_gateup(int R, const StreamParams& p, int ctas, int warps, size_t smem, cudaStream_t s) {
    switch (R) {
        case 1: return launch_stream_instance<kFmtQ4, 2, 1>(p, ctas, warps, smem, s);
        case 2: return launch_stream_instance<kFmtQ4, 2, 2>(p, ctas, warps, smem, s);
        case 4: return launch_stream_instance<kFmtQ4, 2, 4>(p, ctas, warps, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_stream_gateup(int R, size_t smem) {
    switch (R) {
        case 1: return prepare_stream_instance<kFmtQ4, 2, 1>(smem);
        case 2: return prepare_stream_instance<kFmtQ4, 2, 2>(smem);
        case 4: return prepare_stream_instance<kFmtQ4, 2, 4>(smem);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qbw
