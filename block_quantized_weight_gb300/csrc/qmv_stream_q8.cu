// qmv_stream_q8.cu -- instantiations of the streaming M = 1 kernel for Q8_0 (one matrix).
// Split into its own translation unit so the build compiles the variants in parallel.
#include "qmv_stream.cuh"

namespace qbw {

cudaError_t launch_stream_q8(int R, const StreamParams& p, int ctas, int warps, size_t smem, cudaStream_t s) {
    switch (R) {
        case 1: return launch_stream_instance<kFmtQ8, 1, 1>(p, ctas, warps, smem, s);
        case 2: return launch_stream_instance<kFmtQ8, 1, 2>(p, ctas, warps, smem, s);
        case 4: return launch_stream_instance<kFmtQ8, 1, 4>(p, ctas, warps, smem, s);
        case 8: return launch_stream_instance<kFmtQ8, 1, 8>(p, ctas, warps, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_stream_q8(int R, size_t smem) {
    switch (R) {
        case 1: return prepare_stream_instance<kFmtQ8, 1, 1>(smem);
        case 2: return prepare_stream_instance<kFmtQ8, 1, 2>(smem);
        case 4: return prepare_stream_instance<kFmtQ8, 1, 4>(smem);
        case 8: return prepare_stream_instance<kFmtQ8, 1, 8>(smem);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qbw
