// qbw_internal.h -- host/device shared declarations of the qbw library
// (launch parameters, fault codes and the launch functions of each
// translation unit).  Not installed; the public interface is include/qbw.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace qbw {

enum FaultCode : unsigned int {
    kFaultBulkWaitTimeout = 1,   // an mbarrier guarding a bulk copy never completed
    kFaultMmaWaitTimeout = 2,    // an mbarrier guarding tensor-core work never completed
};

enum : int { kFmtQ8 = 0, kFmtQ4 = 1 };

// Launch parameters of the streaming M = 1 kernel (qmv_stream.cuh).
struct StreamParams {
    const uint8_t* w0;     // weights (gate matrix for gate+up)
    const uint8_t* w1;     // up matrix (gate+up only)
    const void* x;         // activations [K]
    void* y;               // outputs [N]
    unsigned int* fault;   // library fault word of this device
    int64_t row_bytes;     // K/32 * block bytes
    int32_t N;
    int32_t K;
    int32_t npairs;        // K/64
    int32_t ntasks;        // ceil(N / R)
    int32_t nfull;         // full 64-block chunks per row (npairs / 32)
    int32_t tail_pairs;    // npairs % 32
    int32_t depth;         // ring stages per warp
    int32_t x_bf16;        // activations are bf16 (else fp32)
    int32_t y_bf16;        // outputs are bf16 (else fp32)
    uint32_t ring_off;     // byte offsets inside dynamic shared memory
    uint32_t bar_off;
    uint32_t stage_bytes;  // NMAT * R * chunk bytes
};

// Block-pair geometry of the streaming kernel.
constexpr int pair_bytes(int fmt) { return fmt == kFmtQ4 ? 36 : 68; }
constexpr int chunk_bytes(int fmt) { return 32 * pair_bytes(fmt); }
constexpr int block_bytes(int fmt) { return fmt == kFmtQ4 ? 18 : 34; }

// Each returns the cudaError_t of the launch (cudaGetLastError after it).
cudaError_t launch_qmv_stream(int fmt, int nmat, int R, const StreamParams& p, int ctas, int warps,
                              size_t smem, cudaStream_t stream);
cudaError_t launch_qmv_generic(int fmt, int nmat, const uint8_t* w0, const uint8_t* w1, const void* x,
                               int x_bf16, void* y, int y_bf16, int64_t N, int64_t K, int sm_count,
                               cudaStream_t stream);
cudaError_t launch_dequant(int fmt, const uint8_t* w, float* out, int64_t N, int64_t K, int sm_count,
                           cudaStream_t stream);

// Largest dynamic shared memory the streaming kernels may request.
cudaError_t prepare_qmv_stream(int fmt, int nmat, int R, size_t smem);

}  // namespace qbw
