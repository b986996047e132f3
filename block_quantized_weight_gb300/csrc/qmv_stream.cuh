// qmv_stream.cuh -- the M = 1 block-quantized matrix-vector kernel (Q8_0,
// Q4_0, and the fused Q4_0 gate+up with GELU-tanh), streaming weight rows from
// HBM through shared memory with 1-D bulk asynchronous copies.
//
// Work decomposition (one persistent CTA per SM, W warps per CTA):
//  * a "task" is R consecutive output rows (R rows of each matrix for
//    gate+up).  Warp g of P takes tasks g, g+P, g+2P, ...;
//  * each task streams its rows in chunks of 64 blocks (32 block pairs); a warp
//    keeps a private ring of D stages, lane 0 issues the bulk copies for the
//    stage D ahead and every lane waits on that stage's mbarrier;
//  * lane l owns block pair l of the chunk for all rows of the task, so the
//    activation slice it needs is loaded from shared memory once and reused
//    R times (the gem decode path's "four-output-row" reuse, generalised);
//  * a final chunk shorter than 64 blocks (K % 2048 != 0) is spread over
//    (row, pair) items so every lane still has work.
//
// A block pair is 36 bytes (Q4_0) or 68 bytes (Q8_0): 4-byte aligned, and its
// internal byte layout is the same for every lane, so all word positions,
// nibble positions and scale positions are compile-time constants.  Lanes read
// 32-bit words at a 9- or 17-word stride: conflict-free across the warp.
//
// Code -> fp32 without an integer-to-float instruction: a code sitting at bit
// p of a word is masked and OR-ed with the exponent of 2^(23-p), which is the
// float 2^(23-p) + code exactly (p = 16 gives 128 + code); one packed fp32x2
// add of -(2^(23-p) + 8) then leaves exactly code - 8, the Q4_0 weight over
// its scale.  Q8_0 bytes are flipped to offset binary (q + 128) inside the
// same LOP3 and the add removes 2^(23-p) + 128, leaving exactly q.  Every
// product code * x is therefore the exact weight-over-scale times x, and a
// block whose weights are all zero contributes exactly zero.
//
// Per block: y += d * sum_j c_j x_j, accumulated in fp32 (packed pairs).
#pragma once

#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"

namespace qbw {

template <int FMT>
struct Fmt;

template <>
struct Fmt<kFmtQ4> {
    static constexpr int kPairBytes = pair_bytes(kFmtQ4);
    static constexpr int kChunkBytes = chunk_bytes(kFmtQ4);
};

template <>
struct Fmt<kFmtQ8> {
    static constexpr int kPairBytes = pair_bytes(kFmtQ8);
    static constexpr int kChunkBytes = chunk_bytes(kFmtQ8);
};

// ---------------------------------------------------------------- slot order
// Each pair's 64 activations are stored in "slot" order: 16 chunks of 4 fp32,
// the order in which the kernel produces decoded codes.
//
// Q4_0 pair words (36 bytes): V0 = [dA, qsA0, qsA1], V1..V3 = qsA[2..13],
// V4 = [qsA14, qsA15, dB], V5..V8 = qsB[0..15].  A word holding qs bytes
// j..j+3 of block X gives two chunks:
//   L: codes at bits 0, 4, 8, 12          -> X(j), X(16+j), X(j+1), X(17+j)
//   H: codes at bits 20, 24, 16, 28       -> X(18+j), X(j+3), X(j+2), X(19+j)
// Chunk 0 = H(V0) (qs bytes 0, 1 at the top of the word, i.e. j = -2),
// chunks 1..6 = L,H of V1..V3, chunk 7 = L(V4) (j = 14), chunks 8..15 = L,H
// of V5..V8.
__host__ __device__ constexpr int q4_chunk_word(int c) {
    return c == 0 ? 0 : (c == 7 ? 4 : (c < 7 ? 1 + (c - 1) / 2 : 5 + (c - 8) / 2));
}
__host__ __device__ constexpr bool q4_chunk_is_h(int c) {
    return c == 0 || (c != 7 && (c < 7 ? (c - 1) % 2 == 1 : (c - 8) % 2 == 1));
}
__host__ __device__ constexpr bool q4_chunk_loads_word(int c) {
    return c == 0 || c == 7 || (c < 7 ? (c - 1) % 2 == 0 : (c - 8) % 2 == 0);
}

// Element (0..63) of the pair multiplied by slot `slot`.
__host__ __device__ constexpr int q4_slot_element(int slot) {
    const int c = slot >> 2, i = slot & 3;
    const int w = q4_chunk_word(c);
    const int blk = (c >= 8) ? 1 : 0;
    const int j0 = (c == 0) ? -2 : (blk ? 4 * (w - 5) : 4 * w - 2);
    int e = 0;
    if (!q4_chunk_is_h(c)) e = (i == 0) ? j0 : (i == 1) ? 16 + j0 : (i == 2) ? j0 + 1 : 17 + j0;
    else e = (i == 0) ? 18 + j0 : (i == 1) ? j0 + 3 : (i == 2) ? j0 + 2 : 19 + j0;
    return blk * 32 + e;
}

// Q8_0 pair words (68 bytes): V0 = [dA, qA0, qA1], V1..V7 = qA[2..29],
// V8 = [qA30, qA31, dB], V9..V16 = qB[0..31].  Chunk 0 = bytes 2,3 of V0 and
// bytes 0,1 of V8; chunk c = 1..7 = the four bytes of Vc; chunk c = 8..15 =
// the four bytes of V(c+1), in memory order.
__host__ __device__ constexpr int q8_slot_element(int slot) {
    const int c = slot >> 2, i = slot & 3;
    if (c == 0) return (i == 0) ? 0 : (i == 1) ? 1 : (i == 2) ? 30 : 31;
    if (c < 8) return 4 * c - 2 + i;
    return 32 + 4 * (c - 8) + i;
}

// ---------------------------------------------------------------- decode
__device__ __forceinline__ uint32_t lop3_select(uint32_t a, uint32_t b, uint32_t c) {
    // per bit: c ? (a ^ b) : b
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6C;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Q4_0 L chunk of word v: codes at bits 0, 4, 8, 12 -> exact (code - 8).
__device__ __forceinline__ void q4_chunk_L(uint32_t v, uint64_t& fa, uint64_t& fb) {
    const uint64_t k01 = 0xC9000080CB000008ull;   // (-(2^23 + 8), -(2^19 + 8))
    const uint64_t k23 = 0xC5008000C7000800ull;   // (-(2^15 + 8), -(2^11 + 8))
    fa = fadd2(pack2((v & 0x0000000Fu) | 0x4B000000u, (v & 0x000000F0u) | 0x49000000u), k01);
    fb = fadd2(pack2((v & 0x00000F00u) | 0x47000000u, (v & 0x0000F000u) | 0x45000000u), k23);
}

// Q4_0 H chunk of word v: codes at bits 20, 24 (shifted to 8, 12) and 16, 28
// (16 in place, 28 shifted to 16) -> exact (code - 8).
__device__ __forceinline__ void q4_chunk_H(uint32_t v, uint64_t& fa, uint64_t& fb) {
    const uint64_t k23 = 0xC5008000C7000800ull;   // (-(2^15 + 8), -(2^11 + 8))
    const uint64_t k16 = 0xC3080000C3080000ull;   // (-(128 + 8), -(128 + 8))
    const uint32_t s = v >> 12;
    fa = fadd2(pack2((s & 0x00000F00u) | 0x47000000u, (s & 0x0000F000u) | 0x45000000u), k23);
    fb = fadd2(pack2((v & 0x000F0000u) | 0x43000000u, (s & 0x000F0000u) | 0x43000000u), k16);
}

// Q8_0: the signed bytes 0 and 1 of word v -> exact floats.
__device__ __forceinline__ uint64_t q8_bytes01(uint32_t v) {
    const uint64_t k = 0xC7008000CB000080ull;     // (-(2^23 + 128), -(2^15 + 128))
    const uint32_t a = lop3_select(v, 0x4B000080u, 0x000000FFu);   // 2^23 + (q0 + 128)
    const uint32_t b = lop3_select(v, 0x47008000u, 0x0000FF00u);   // 2^15 + (q1 + 128)
    return fadd2(pack2(a, b), k);
}

// ---------------------------------------------------------------- one pair
// Accumulate one block pair of NR rows of NMAT matrices into acc.
// rowaddr(m, r) is the shared-memory address of the pair in row (m, r).
template <int FMT, int NMAT, int NR, typename RowAddr>
__device__ __forceinline__ void pair_dot(const RowAddr& rowaddr, uint32_t xaddr, uint32_t swz,
                                         float (&acc)[NMAT][NR]) {
    uint64_t bacc[NMAT][NR];
    uint32_t vw[NMAT][NR];
    uint32_t dA[NMAT][NR], dB[NMAT][NR];
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < NR; ++r) { bacc[m][r] = 0ull; vw[m][r] = 0u; dA[m][r] = 0u; dB[m][r] = 0u; }

#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float4 xv = lds128f(xaddr + (((uint32_t)c ^ swz) << 4));
        const uint64_t x01 = pack2f(xv.x, xv.y);
        const uint64_t x23 = pack2f(xv.z, xv.w);
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t base = rowaddr(m, r);
                uint64_t fa, fb;
                if constexpr (FMT == kFmtQ4) {
                    if (q4_chunk_loads_word(c)) vw[m][r] = lds32(base + 4u * (uint32_t)q4_chunk_word(c));
                    const uint32_t v = vw[m][r];
                    if (c == 0) dA[m][r] = v;
                    if (c == 7) dB[m][r] = v >> 16;
                    if (q4_chunk_is_h(c)) q4_chunk_H(v, fa, fb);
                    else q4_chunk_L(v, fa, fb);
                } else {
                    if (c == 0) {
                        const uint32_t v0 = lds32(base);
                        const uint32_t v8 = lds32(base + 32u);
                        dA[m][r] = v0;
                        dB[m][r] = v8 >> 16;
                        fa = q8_bytes01(v0 >> 16);
                        fb = q8_bytes01(v8);
                    } else {
                        const uint32_t v = lds32(base + 4u * (uint32_t)((c < 8) ? c : c + 1));
                        fa = q8_bytes01(v);
                        fb = q8_bytes01(v >> 16);
                    }
                }
                ffma2(bacc[m][r], fa, x01);
                ffma2(bacc[m][r], fb, x23);
                if (c == 7 || c == 15) {
                    const float2 s = unpack2f(bacc[m][r]);
                    const float t = s.x + s.y;
                    const float d = half_bits_to_float(c == 7 ? dA[m][r] : dB[m][r]);
                    acc[m][r] = fmaf(d, t, acc[m][r]);
                    bacc[m][r] = 0ull;
                }
            }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Stage the activations in slot order: 64 fp32 per pair, 16-byte chunks
// XOR-swizzled by pair index so that 8 lanes reading 8 consecutive pairs hit 8
// distinct bank groups.
template <int FMT>
__device__ __forceinline__ void stage_activations(const StreamParams& p, uint8_t* smem) {
    float* xs = reinterpret_cast<float*>(smem);
    for (int q = threadIdx.x; q < p.npairs; q += blockDim.x) {
        const uint32_t swz = (uint32_t)q & 7u;
#pragma unroll 4
        for (int s = 0; s < 64; ++s) {
            const int e = (FMT == kFmtQ4) ? q4_slot_element(s) : q8_slot_element(s);
            const int64_t k = (int64_t)q * 64 + e;
            const float xv = p.x_bf16 ? load_act<__nv_bfloat16>(p.x, k) : load_act<float>(p.x, k);
            xs[q * 64 + (int)((((uint32_t)(s >> 2)) ^ swz) << 2) + (s & 3)] = xv;
        }
    }
}

// ---------------------------------------------------------------- the kernel
template <int FMT, int NMAT, int R>
__global__ void __launch_bounds__(512, 1) qmv_stream_kernel(const StreamParams p) {
    using F = Fmt<FMT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int gw = blockIdx.x * nwarps + warp;
    const int P = gridDim.x * nwarps;
    const int D = p.depth;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t xs = sbase;                                    // 64 fp32 per pair
    const uint32_t ring = sbase + p.ring_off + (uint32_t)warp * (uint32_t)D * p.stage_bytes;
    const uint32_t bars = sbase + p.bar_off + (uint32_t)warp * (uint32_t)D * 8u;

    const int nitems = p.nfull + (p.tail_pairs ? 1 : 0);
    const int my_tasks = (p.ntasks > gw) ? (p.ntasks - gw + P - 1) / P : 0;
    const int total = my_tasks * nitems;
    const uint64_t policy = policy_evict_first();

    // Lane 0 only: copy item j (task j / nitems, chunk j % nitems) into stage j % D.
    auto issue = [&](int j) {
        const int ti = j / nitems, c = j - ti * nitems;
        const int64_t row0 = (int64_t)(gw + ti * P) * R;
        const int64_t left = (int64_t)p.N - row0;
        const int rows = left < R ? (int)left : R;
        const uint32_t bytes = (c < p.nfull) ? (uint32_t)F::kChunkBytes
                                             : (uint32_t)(p.tail_pairs * F::kPairBytes);
        const int s = j % D;
        const uint32_t bar = bars + 8u * (uint32_t)s;
        const uint32_t dst0 = ring + (uint32_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(bar, bytes * (uint32_t)(rows * NMAT));
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            const uint8_t* wm = (m == 0) ? p.w0 : p.w1;
            for (int r = 0; r < rows; ++r) {
                const uint8_t* src = wm + (row0 + r) * p.row_bytes + (int64_t)c * F::kChunkBytes;
                bulk_g2s(dst0 + (uint32_t)(m * R + r) * (uint32_t)F::kChunkBytes, src, bytes, bar, policy);
            }
        }
    };

    if (lane == 0) {
        for (int s = 0; s < D; ++s) mbar_init(bars + 8u * (uint32_t)s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (lane == 0)
        for (int j = 0; j < min(D, total); ++j) issue(j);

    stage_activations<FMT>(p, smem);
    __syncthreads();

    float acc[NMAT][R];
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[m][r] = 0.f;

    int j = 0;
    for (; j < total; ++j) {
        const int s = j % D;
        const uint32_t parity = (uint32_t)(j / D) & 1u;
        const bool arrived = mbar_wait_bounded(bars + 8u * (uint32_t)s, parity, p.fault, kFaultBulkWaitTimeout);
        if (!__all_sync(0xffffffffu, arrived)) break;

        const int ti = j / nitems, c = j - ti * nitems;
        const int64_t row0 = (int64_t)(gw + ti * P) * R;
        const uint32_t stage = ring + (uint32_t)s * p.stage_bytes;
        if (c < p.nfull) {
            const int q = c * 32 + lane;
            const uint32_t poff = (uint32_t)lane * (uint32_t)F::kPairBytes;
            auto rowaddr = [&](int m, int r) {
                return stage + (uint32_t)(m * R + r) * (uint32_t)F::kChunkBytes + poff;
            };
            pair_dot<FMT, NMAT, R>(rowaddr, xs + (uint32_t)q * 256u, (uint32_t)q & 7u, acc);
        } else {
            // tail chunk: (row, pair) items spread over the lanes
            const int items = R * p.tail_pairs;
            for (int it = lane; it < items; it += 32) {
                const int r = it / p.tail_pairs;
                const int qq = it - r * p.tail_pairs;
                const int q = c * 32 + qq;
                float part[NMAT][1];
#pragma unroll
                for (int m = 0; m < NMAT; ++m) part[m][0] = 0.f;
                auto rowaddr = [&](int m, int) {
                    return stage + (uint32_t)(m * R + r) * (uint32_t)F::kChunkBytes +
                           (uint32_t)qq * (uint32_t)F::kPairBytes;
                };
                pair_dot<FMT, NMAT, 1>(rowaddr, xs + (uint32_t)q * 256u, (uint32_t)q & 7u, part);
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr)
                        if (rr == r) acc[m][rr] += part[m][0];
            }
        }
        __syncwarp();
        if (lane == 0 && j + D < total) {
            fence_proxy_async_smem();
            issue(j + D);
        }
        if (c == nitems - 1) {
            float outv = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float g = warp_sum(acc[0][r]);
                float v = g;
                if constexpr (NMAT == 2) {
                    const float u = warp_sum(acc[1][r]);
                    v = gelu_tanh(g) * u;
                }
                if (lane == r) outv = v;
            }
            if (lane < R && row0 + lane < p.N) {
                if (p.y_bf16) store_out<__nv_bfloat16>(p.y, row0 + lane, outv);
                else store_out<float>(p.y, row0 + lane, outv);
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int r = 0; r < R; ++r) acc[m][r] = 0.f;
        }
    }
    if (j < total && lane == 0) {
        // A copy never arrived.  Before leaving, give the other stages already
        // in flight the same bounded time to land in this CTA's shared memory.
        for (int jj = j + 1; jj < min(total, j + D); ++jj)
            mbar_wait_bounded(bars + 8u * (uint32_t)(jj % D), (uint32_t)(jj / D) & 1u, p.fault,
                              kFaultBulkWaitTimeout);
    }
}

// Host-side launch of one instantiation.
template <int FMT, int NMAT, int R>
cudaError_t launch_stream_instance(const StreamParams& p, int ctas, int warps, size_t smem,
                                   cudaStream_t stream) {
    qmv_stream_kernel<FMT, NMAT, R><<<ctas, warps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int FMT, int NMAT, int R>
cudaError_t prepare_stream_instance(size_t smem) {
    return cudaFuncSetAttribute(qmv_stream_kernel<FMT, NMAT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
}

}  // namespace qbw
