// qbw_internal.h -- host/device shared declarations of the qbw library
// (launch parameters, fault codes and the launch functions of each
// translation unit).  Not installed; the public interface is include/qbw.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace qbw {

enum FaultCode : unsigned int {
    kFaultBulkWaitTimeout = 1,   // an mbarrier guarding a bulk copy never completed
    kFaultMmaWaitTimeout = 2,    // an mbarrier guarding tensor-core work never completed
    kFaultBadIndex = 3,          // a token-table row index outside [0, N)
    kFaultShareWaitTimeout = 4,  // a split tile's share from another CTA never arrived
    kFaultPlan = 5,              // a launch plan exceeded a kernel's fixed capacity (internal)
    kFaultGridWait = 6,          // a chain's CTAs waited in vain for the others between steps
};

// kFmtMix4, kFmtMix2, kFmtMix8: the int4-affine, int2-symmetric and int8
// mixed-bit matrices with groups of 32 (codes, scales and, for int4, biases in
// their own arrays), on the tensor-core M = 1 kernel only
enum : int { kFmtQ8 = 0, kFmtQ4 = 1, kFmtQ4K = 2, kFmtMix4 = 3, kFmtMix2 = 4, kFmtMix8 = 5 };

// Bytes of one row of K weights: Q8_0 34 and Q4_0 18 per 32 weights; Q4_K
// 144 per 256-weight super-block.
constexpr int64_t weight_row_bytes(int fmt, int64_t K) {
    return fmt == kFmtQ4K ? (K / 256) * 144 : (K / 32) * (fmt == kFmtQ4 ? 18 : 34);
}

// Launch parameters of the streaming M = 1 kernel (qmv_stream.cuh).
// tmap[m] views weight matrix m as a 2-D array of 8-byte elements,
// [N rows][row_bytes / 8], with a box of (chunk or half-chunk) x R rows.
struct StreamParams {
    CUtensorMap tmap[2];   // weights (gate, up for gate+up)
    const uint8_t* w0;     // weights (gate matrix for gate+up)
    const uint8_t* w1;     // up matrix (gate+up only)
    const void* x;         // activations [K]
    void* y;               // outputs [N]
    unsigned int* fault;   // library fault word of this device
    int64_t row_bytes;     // K/32 * block bytes
    int32_t N;
    int32_t K;
    int32_t npairs;        // K/64
    int32_t ngroups;       // row groups of R rows: ceil(N / R)
    int32_t nfull;         // full 64-block chunks per row (npairs / 32)
    int32_t tail_pairs;    // npairs % 32
    int32_t depth;         // ring stages per warp
    int32_t x_bf16;        // activations are bf16 (else fp32)
    int32_t x_vec;         // x is aligned for 4-element vector loads (16 B fp32, 8 B bf16)
    int32_t y_bf16;        // outputs are bf16 (else fp32)
    uint32_t ring_off;     // byte offsets inside dynamic shared memory
    uint32_t bar_off;
    uint32_t part_off;     // per-item row partials (fp32)
    uint32_t slot_off;     // 64-byte table: slot of each pair element
    uint32_t stage_bytes;  // bytes of one ring stage (all matrices, all rows)
    uint32_t mat_bytes;    // bytes of one matrix's rows within a stage
    uint32_t half_bytes;   // Q8_0: bytes of one half-chunk box (R rows), 128-aligned
};

// Block-pair geometry of the streaming kernel.
constexpr int pair_bytes(int fmt) { return fmt == kFmtQ4 ? 36 : 68; }
constexpr int chunk_bytes(int fmt) { return 32 * pair_bytes(fmt); }
constexpr int block_bytes(int fmt) { return fmt == kFmtQ4 ? 18 : 34; }
// Tensor-copy boxes per chunk: Q4_0 one box of 144 8-byte words (1152 bytes);
// Q8_0 two boxes of 136 words (1088 bytes, 16 pairs each), as a box row may
// hold at most 256 elements.
constexpr int boxes_per_chunk(int fmt) { return fmt == kFmtQ4 ? 1 : 2; }
constexpr int box_words(int fmt) { return fmt == kFmtQ4 ? 144 : 136; }
constexpr int pairs_per_box(int fmt) { return fmt == kFmtQ4 ? 32 : 16; }
// Shared-memory layout of one ring stage: per matrix, per box, R rows of
// box_words * 8 bytes; every box starts on a 128-byte boundary.
constexpr uint32_t stage_half_bytes(int fmt, int R) { return (uint32_t)((R * box_words(fmt) * 8 + 127) / 128 * 128); }
constexpr uint32_t stage_mat_bytes(int fmt, int R) { return stage_half_bytes(fmt, R) * boxes_per_chunk(fmt); }
constexpr uint32_t stage_bytes_of(int fmt, int nmat, int R) { return stage_mat_bytes(fmt, R) * nmat; }

// Each returns the cudaError_t of the launch (cudaGetLastError after it).
cudaError_t launch_qmv_stream(int fmt, int nmat, int R, const StreamParams& p, int ctas, int warps,
                              size_t smem, cudaStream_t stream);
cudaError_t launch_qmv_generic(int fmt, int nmat, const uint8_t* w0, const uint8_t* w1, const void* x,
                               int x_bf16, void* y, int y_bf16, int64_t N, int64_t K, int sm_count,
                               cudaStream_t stream);
cudaError_t launch_dequant(int fmt, const uint8_t* w, float* out, int64_t N, int64_t K, int sm_count,
                           cudaStream_t stream);
cudaError_t launch_embed(int fmt, const uint8_t* w, const int32_t* ids, int64_t n_ids, int64_t N, int64_t K, void* out,
                         int out_bf16, unsigned int* fault, int sm_count, cudaStream_t stream);

// qmv_mixbit.cu: the mixed-bit (2-, 4-, 8-bit) matrix-vector product and its
// dequantizer.  x is staged in shared memory beside the warps' copy rings:
// qmv_mixbit_smem_bytes(bits, K, group) must not exceed kMixMaxSmem.
constexpr size_t kMixMaxSmem = 227 * 1024;
size_t qmv_mixbit_smem_bytes(int bits, int64_t K, int64_t group);
cudaError_t launch_qmv_mixbit(int bits, const void* qp, const void* sc, const void* bi, int G, const void* x,
                              int x_bf16, void* y, int y_bf16, int N, int K, int sm_count, cudaStream_t stream);
cudaError_t launch_dequant_mixbit(int bits, const void* qp, const void* sc, const void* bi, int G, float* out, int N,
                                  int K, int sm_count, cudaStream_t stream);

// qmm_noalloc.cu: the next qmm_q4_0_smallM_noalloc call on `device` zero-fills
// its static scratch again (called when qbw_fault_read finds a fault).
void noalloc_scratch_mark_dirty(int device);

// Largest dynamic shared memory the streaming kernels may request.
cudaError_t prepare_qmv_stream(int fmt, int nmat, int R, size_t smem);

// The launch after a tensor-core M = 1 launch on the same stream, for the
// L2 prefetch of its first weight tiles: its tensor maps (the up matrix in
// [1] for gate+up) and unit split (units = tiles x groups x nmat).
struct QtcNextLaunch {
    CUtensorMap tmap[2];
    int32_t units, groups, nmat;
};

// One step of a chained product (qmv_chain.cu), in device memory (aligned as
// its tensor maps require): y = W x (nmat = 1) or gelu_tanh(Wg x) * (Wu x)
// (nmat = 2), Q4_0 weights, bf16 x.
struct ChainStepDesc {
    CUtensorMap tmap[2];      // the (gate) matrix and, for nmat = 2, the up matrix
    const void* x;            // bf16 [K]
    void* y;                  // [N], bf16 (y_bf16) or fp32
    const uint8_t* w[2];      // the raw weights of tmap[0], tmap[1] (the read-back correction reads a row)
    int32_t N, K, nmat, y_bf16;
    int32_t tiles, groups, units, reserved;
};

}  // namespace qbw
