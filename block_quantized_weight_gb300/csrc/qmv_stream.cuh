// qmv_stream.cuh -- the M = 1 block-quantized matrix-vector kernel (Q8_0,
// Q4_0, and the fused Q4_0 gate+up with GELU-tanh), streaming weight rows from
// HBM through shared memory with 1-D bulk asynchronous copies.
//
// Work decomposition (one persistent CTA per SM, W warps per CTA):
//  * rows form groups of R consecutive rows (R rows of each matrix for
//    gate+up); each CTA owns a contiguous range of groups;
//  * a row is cut into chunks of 64 blocks (32 block pairs); the CTA's work
//    items are (group, chunk) pairs, dealt round-robin to its warps, so the
//    items of one group run on different warps at the same time;
//  * each warp keeps a private ring of D shared-memory stages: lane 0 issues
//    the bulk copies of the item D ahead, every lane waits on that stage's
//    mbarrier (bounded wait);
//  * within an item, lane l owns block pair l of the chunk for all R rows, so
//    the activation slice it needs is read from shared memory once and reused
//    R times (the gem decode path's "four-output-row" reuse, generalised);
//    a final chunk shorter than 64 blocks is spread over (row, pair) items;
//  * each item's R row partials are reduced across the warp and stored in
//    shared memory; at the end the CTA adds every row's partials in chunk
//    order (a fixed order: results are bit-reproducible) and writes y.
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
// Exponent fields of 2^23, 2^19, 2^15, 2^11, 2^7: OR-ed above a code sitting at
// bit 0, 4, 8, 12, 16 they make the float 2^e + code.
constexpr uint32_t kMag23 = 0x4B000000u, kMag19 = 0x49000000u, kMag15 = 0x47000000u, kMag11 = 0x45000000u,
                   kMag7 = 0x43000000u;
// Packed (lo, hi) fp32 constants subtracted after the OR: -(2^e + 8) for Q4_0.
constexpr uint64_t kSubQ4_23_19 = 0xC9000080CB000008ull;   // (-(2^23 + 8), -(2^19 + 8))
constexpr uint64_t kSubQ4_15_11 = 0xC5008000C7000800ull;   // (-(2^15 + 8), -(2^11 + 8))
constexpr uint64_t kSubQ4_7_7 = 0xC3080000C3080000ull;     // (-(2^7 + 8), -(2^7 + 8))
// Q8_0: -(2^e + 128) undoes the magic and the offset-binary flip.
constexpr uint64_t kSubQ8 = 0xC7008000CB000080ull;         // (-(2^23 + 128), -(2^15 + 128))

// Two codes -> one fp32x2 register pair, in one asm block so that the two
// LOP3 results land directly in the pair the packed add reads:
//   lo = (a & ML) | gl,  hi = (b & MH) | gh,  result = (lo, hi) + k.
template <uint32_t ML, uint32_t MH>
__device__ __forceinline__ uint64_t codes2(uint32_t a, uint32_t b, uint32_t gl, uint32_t gh, uint64_t k) {
    uint64_t r;
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 t;\n\t"
        "lop3.b32 lo, %1, %5, %3, 0xEA;\n\t"
        "lop3.b32 hi, %2, %6, %4, 0xEA;\n\t"
        "mov.b64 t, {lo, hi};\n\t"
        "add.rn.f32x2 %0, t, %7;\n\t}"
        : "=l"(r)
        : "r"(a), "r"(b), "r"(gl), "r"(gh), "n"(ML), "n"(MH), "l"(k));
    return r;
}

// Q8_0: bytes at bits 0 and 8 of a and b, signed -> (q_lo, q_hi) exactly.
// Per bit: mask ? (v ^ g) : g, with g = exponent | 0x80 flip bit (LOP3 0x6C).
__device__ __forceinline__ uint64_t q8_codes2(uint32_t a, uint32_t b, uint32_t gl, uint32_t gh) {
    uint64_t r;
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 t;\n\t"
        "lop3.b32 lo, %1, %3, 0x000000FF, 0x6C;\n\t"
        "lop3.b32 hi, %2, %4, 0x0000FF00, 0x6C;\n\t"
        "mov.b64 t, {lo, hi};\n\t"
        "add.rn.f32x2 %0, t, %5;\n\t}"
        : "=l"(r)
        : "r"(a), "r"(b), "r"(gl), "r"(gh), "l"(kSubQ8));
    return r;
}

// Register-resident magic constants (materialised once per thread).
struct Mags {
    uint32_t m23, m19, m15, m11, m7, q8a, q8b;
    __device__ __forceinline__ Mags()
        : m23(kMag23), m19(kMag19), m15(kMag15), m11(kMag11), m7(kMag7), q8a(0x4B000080u), q8b(0x47008000u) {}
};

// Q4_0 L chunk of word v: codes at bits 0, 4, 8, 12 -> exact (code - 8).
__device__ __forceinline__ void q4_chunk_L(uint32_t v, const Mags& g, uint64_t& fa, uint64_t& fb) {
    fa = codes2<0x0000000Fu, 0x000000F0u>(v, v, g.m23, g.m19, kSubQ4_23_19);
    fb = codes2<0x00000F00u, 0x0000F000u>(v, v, g.m15, g.m11, kSubQ4_15_11);
}

// Q4_0 H chunk of word v: codes at bits 20, 24 (shifted down by 12 to 8, 12)
// and at bits 16 (in place) and 28 (shifted to 16) -> exact (code - 8).
__device__ __forceinline__ void q4_chunk_H(uint32_t v, const Mags& g, uint64_t& fa, uint64_t& fb) {
    const uint32_t s = v >> 12;
    fa = codes2<0x00000F00u, 0x0000F000u>(s, s, g.m15, g.m11, kSubQ4_15_11);
    fb = codes2<0x000F0000u, 0x000F0000u>(v, s, g.m7, g.m7, kSubQ4_7_7);
}

// ---------------------------------------------------------------- one pair
// Accumulate one block pair of NR rows of NMAT matrices into acc.
// rowaddr(m, r) is the shared-memory address of the pair in row (m, r); xaddr
// the pair's 16 chunks of 4 activations.  Block A (chunks 0..7) of every row,
// then block B (chunks 8..15): each row loads only the words of the block at
// hand, and the scale is a half of one of them.
template <int FMT, int NMAT, int NR, typename RowAddr>
__device__ __forceinline__ void pair_dot(const RowAddr& rowaddr, uint32_t xaddr, const Mags& g,
                                         float (&acc)[NMAT][NR]) {
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint64_t xv[8][2];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 f = lds128f(xaddr + 16u * (uint32_t)(8 * blk + k));
            xv[k][0] = pack2f(f.x, f.y);
            xv[k][1] = pack2f(f.z, f.w);
        }
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint32_t base = rowaddr(m, r);
                uint64_t bacc = 0ull;
                uint32_t dbits;
                if constexpr (FMT == kFmtQ4) {
                    // block A: V0 (hi half), V1..V3, V4 (lo half); block B: V5..V8, dB in V4's hi half
                    uint32_t v[5];
#pragma unroll
                    for (int i = 0; i < 5; ++i) v[i] = lds32(base + 4u * (uint32_t)(blk == 0 ? i : 4 + i));
                    dbits = (blk == 0) ? v[0] : (v[0] >> 16);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int c = 8 * blk + k;
                        const uint32_t w = v[q4_chunk_word(c) - (blk == 0 ? 0 : 4)];
                        uint64_t fa, fb;
                        if (q4_chunk_is_h(c)) q4_chunk_H(w, g, fa, fb);
                        else q4_chunk_L(w, g, fa, fb);
                        ffma2(bacc, fa, xv[k][0]);
                        ffma2(bacc, fb, xv[k][1]);
                    }
                } else {
                    // block A: V0 (hi half), V1..V7, V8 (lo half); block B: V9..V16, dB in V8's hi half
                    uint32_t v[9];
#pragma unroll
                    for (int i = 0; i < 9; ++i) v[i] = lds32(base + 4u * (uint32_t)(blk == 0 ? i : 8 + i));
                    dbits = (blk == 0) ? v[0] : (v[0] >> 16);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint64_t fa, fb;
                        if (blk == 0 && k == 0) {
                            const uint32_t h0 = v[0] >> 16;
                            fa = q8_codes2(h0, h0, g.q8a, g.q8b);
                            fb = q8_codes2(v[8], v[8], g.q8a, g.q8b);
                        } else {
                            const uint32_t w = v[blk == 0 ? k : k + 1];
                            const uint32_t h = w >> 16;
                            fa = q8_codes2(w, w, g.q8a, g.q8b);
                            fb = q8_codes2(h, h, g.q8a, g.q8b);
                        }
                        ffma2(bacc, fa, xv[k][0]);
                        ffma2(bacc, fb, xv[k][1]);
                    }
                }
                const float2 sv = unpack2f(bacc);
                acc[m][r] = fmaf(half_bits_to_float(dbits), sv.x + sv.y, acc[m][r]);
            }
    }
}

// Activations of one pair in shared memory: 64 fp32 in slot order, padded to
// 68 (272 bytes, 17 bank groups of 16 bytes), so 8 lanes reading the same
// chunk of 8 consecutive pairs hit 8 distinct bank groups.
constexpr int kXsPairFloats = 68;

// Stage the activations in slot order.  slot_of[e] is the slot of pair element
// e (filled by the caller).  Each thread loads groups of 4 consecutive
// elements (vector loads when x is aligned for them): group i of thread t is
// i = t + u * blockDim.  All the loads of the first batch, which covers every
// activation of K up to 4 * kStageBatch * blockDim (21504 at 12 warps), are
// issued before the caller starts the weight copies: loads issued after them
// wait behind a full ring of weight traffic.
constexpr int kStageBatch = 16;

struct StageBatch {
    float v[kStageBatch][4];
};

__device__ __forceinline__ void load_x4(const StreamParams& p, int i, float (&v)[4]) {
    if (p.x_bf16) {
        uint32_t lo, hi;
        if (p.x_vec) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.x) + i);
            lo = raw.x;
            hi = raw.y;
        } else {
            const unsigned short* h = reinterpret_cast<const unsigned short*>(p.x) + 4 * i;
            lo = (uint32_t)__ldg(h) | ((uint32_t)__ldg(h + 1) << 16);
            hi = (uint32_t)__ldg(h + 2) | ((uint32_t)__ldg(h + 3) << 16);
        }
        v[0] = __uint_as_float(lo << 16);
        v[1] = __uint_as_float(lo & 0xFFFF0000u);
        v[2] = __uint_as_float(hi << 16);
        v[3] = __uint_as_float(hi & 0xFFFF0000u);
    } else if (p.x_vec) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p.x) + i);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
        const float* f = reinterpret_cast<const float*>(p.x) + 4 * i;
        v[0] = __ldg(f); v[1] = __ldg(f + 1); v[2] = __ldg(f + 2); v[3] = __ldg(f + 3);
    }
}

__device__ __forceinline__ void load_batch(const StreamParams& p, int i0, StageBatch& bt) {
    const int n4 = p.K >> 2;
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i < n4) load_x4(p, i, bt.v[u]);
    }
}

// Group i covers elements 4 (i % 16) .. +3 of pair i / 16.  blockDim is a
// multiple of 32, so i % 16 is the same for all of a thread's groups and the
// four slots sl[] are looked up once.
__device__ __forceinline__ void store_batch(const StreamParams& p, int i0, const StageBatch& bt, float* xs,
                                            const int (&sl)[4]) {
    const int n4 = p.K >> 2;
#pragma unroll
    for (int u = 0; u < kStageBatch; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i >= n4) break;
        float* q = xs + (i >> 4) * kXsPairFloats;
#pragma unroll
        for (int t = 0; t < 4; ++t) q[sl[t]] = bt.v[u][t];
    }
}

// Finish staging: store the first batch, then load and store the rest.
__device__ __forceinline__ void stage_activations_end(const StreamParams& p, const StageBatch& first, float* xs,
                                                      const uint8_t* slot_of) {
    int sl[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) sl[t] = slot_of[((threadIdx.x & 15) << 2) + t];
    store_batch(p, (int)threadIdx.x, first, xs, sl);
    const int n4 = p.K >> 2;
    for (int i0 = (int)threadIdx.x + kStageBatch * (int)blockDim.x; i0 < n4; i0 += kStageBatch * (int)blockDim.x) {
        StageBatch bt;
        load_batch(p, i0, bt);
        store_batch(p, i0, bt, xs, sl);
    }
}

// Sum V values per lane across the 32 lanes of the warp.  Returns, in every
// lane, the total of value index value_of_lane(lane); the exchange pattern is
// fixed, so the result is bit-reproducible.
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane) {
    int off = 16;
#pragma unroll
    for (int half = V / 2; half >= 1; half /= 2, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float t = v[0];
#pragma unroll
    for (; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return t;
}

// Value index a lane holds after transpose_reduce<V>.
template <int V>
__device__ __forceinline__ int value_of_lane(int lane) {
    int idx = 0, off = 16;
#pragma unroll
    for (int half = V / 2; half >= 1; half /= 2, off >>= 1) idx = (idx << 1) | ((lane & off) ? 1 : 0);
    return idx;
}

// ---------------------------------------------------------------- the kernel
template <int FMT, int NMAT, int R>
__global__ void __launch_bounds__(512, 1) qmv_stream_kernel(const __grid_constant__ StreamParams p) {
    using F = Fmt<FMT>;
    constexpr int V = NMAT * R;                 // row partials per item
    constexpr uint32_t kHalf = stage_half_bytes(FMT, R);
    constexpr uint32_t kMat = stage_mat_bytes(FMT, R);
    constexpr uint32_t kStage = stage_bytes_of(FMT, NMAT, R);
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* slot_of = smem + p.slot_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = blockDim.x >> 5;
    const int D = p.depth;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t xs = sbase;                                    // kXsPairFloats fp32 per pair
    const uint32_t ring = sbase + p.ring_off + (uint32_t)warp * (uint32_t)D * kStage;
    const uint32_t bars = sbase + p.bar_off + (uint32_t)warp * (uint32_t)D * 8u;
    float* part = reinterpret_cast<float*>(smem + p.part_off);

    // this CTA's groups and items
    // groups [g0, g1): ngroups split into gridDim.x near-equal contiguous ranges
    const int gq = p.ngroups / (int)gridDim.x, gr = p.ngroups - gq * (int)gridDim.x;
    const int b = (int)blockIdx.x;
    const int g0 = b * gq + (b < gr ? b : gr);
    const int g1 = g0 + gq + (b < gr ? 1 : 0);
    const int nitems = p.nfull + (p.tail_pairs ? 1 : 0);
    const int n_items = (g1 - g0) * nitems;
    const int mine = (n_items > warp) ? (n_items - warp + W - 1) / W : 0;
    const uint64_t policy = policy_evict_first();

    // Lane 0 only: copy item (group g0 + lg, chunk c) into stage `st` with
    // one tensor copy per matrix and box; rows past N and words past the end
    // of a row arrive as zeros, and every box counts in full.
    auto issue = [&](int lg, int c, int st) {
        const uint32_t bar = bars + 8u * (uint32_t)st;
        const uint32_t dst0 = ring + (uint32_t)st * kStage;
        mbar_arrive_expect_tx(bar, (uint32_t)(NMAT * boxes_per_chunk(FMT) * box_words(FMT) * 8 * R));
        const int y = (g0 + lg) * R;
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int h = 0; h < boxes_per_chunk(FMT); ++h)
                tma_load_2d(dst0 + (uint32_t)m * kMat + (uint32_t)h * kHalf, &p.tmap[m],
                            (c * boxes_per_chunk(FMT) + h) * box_words(FMT), y, bar, policy);
    };

    // the item after (lg, c) for this warp: c advances by W chunks
    const int step_g = W / nitems, step_c = W - (W / nitems) * nitems;
    auto next_item = [&](int& lg_, int& c_) {
        lg_ += step_g;
        c_ += step_c;
        if (c_ >= nitems) { c_ -= nitems; ++lg_; }
    };

    if (lane == 0) {
        for (int s = 0; s < D; ++s) mbar_init(bars + 8u * (uint32_t)s, 1);
        fence_mbar_init();
        prefetch_tmap(&p.tmap[0]);
        if (NMAT == 2) prefetch_tmap(&p.tmap[1]);
    }
    if (threadIdx.x < 64)
        slot_of[FMT == kFmtQ4 ? q4_slot_element(threadIdx.x) : q8_slot_element(threadIdx.x)] = (uint8_t)threadIdx.x;
    __syncwarp();

    // The activations may come from the preceding grid: wait for it, then
    // issue their loads before the weight copies so they are not queued
    // behind them.
    grid_dependency_wait();
    StageBatch first;
    load_batch(p, (int)threadIdx.x, first);

    // producer cursor (lane 0): the item D ahead of the consumer
    int plg = warp / nitems, pc = warp - (warp / nitems) * nitems, pst = 0;
    if (lane == 0)
        for (int j = 0; j < min(D, mine); ++j) {
            issue(plg, pc, pst);
            next_item(plg, pc);
            if (++pst == D) pst = 0;
        }

    __syncthreads();                    // slot table complete
    stage_activations_end(p, first, reinterpret_cast<float*>(smem), slot_of);
    __syncthreads();
    grid_launch_dependents();

    const Mags g;
    // (row, pair) of this lane's first short-chunk item, and the step per 32 items
    const int tail_tp = p.tail_pairs > 0 ? p.tail_pairs : 1;
    const int tail_r0 = lane / tail_tp, tail_q0 = lane - (lane / tail_tp) * tail_tp;
    const int tail_dr = 32 / tail_tp, tail_dq = 32 - (32 / tail_tp) * tail_tp;
    int j = 0, s = 0, lg = warp / nitems, c = warp - (warp / nitems) * nitems;
    uint32_t parity = 0;
    for (; j < mine; ++j) {
        const bool arrived = mbar_wait_bounded(bars + 8u * (uint32_t)s, parity, p.fault, kFaultBulkWaitTimeout);
        if (!__all_sync(0xffffffffu, arrived)) break;

        const int it = lg * nitems + c;
        const uint32_t stage = ring + (uint32_t)s * kStage;
        float acc[NMAT][R];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.f;
        if (c < p.nfull) {
            const int q = c * 32 + lane;
            const uint32_t poff = (FMT == kFmtQ4)
                                      ? (uint32_t)lane * (uint32_t)F::kPairBytes
                                      : (uint32_t)(lane >> 4) * kHalf + (uint32_t)(lane & 15) * F::kPairBytes;
            constexpr uint32_t kRowBytes = (uint32_t)(box_words(FMT) * 8);
            auto rowaddr = [&](int m, int r) {
                return stage + (uint32_t)m * kMat + (uint32_t)r * kRowBytes + poff;
            };
            pair_dot<FMT, NMAT, R>(rowaddr, xs + (uint32_t)q * (4u * kXsPairFloats), g, acc);
        } else {
            // final short chunk: (row, pair) items spread over the lanes
            const int items = R * p.tail_pairs;
            int r = tail_r0, qq = tail_q0;
            for (int t = lane; t < items; t += 32) {
                const int q = c * 32 + qq;
                float one[NMAT][1];
#pragma unroll
                for (int m = 0; m < NMAT; ++m) one[m][0] = 0.f;
                const uint32_t poff = (FMT == kFmtQ4)
                                          ? (uint32_t)qq * (uint32_t)F::kPairBytes
                                          : (uint32_t)(qq >> 4) * kHalf + (uint32_t)(qq & 15) * F::kPairBytes;
                const uint32_t rbase = stage + (uint32_t)r * (uint32_t)(box_words(FMT) * 8) + poff;
                auto rowaddr = [&](int m, int) { return rbase + (uint32_t)m * kMat; };
                pair_dot<FMT, NMAT, 1>(rowaddr, xs + (uint32_t)q * (4u * kXsPairFloats), g, one);
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr)
                        if (rr == r) acc[m][rr] += one[m][0];
                // next item of this lane: t + 32 = (r + tail_dr) rows, (qq + tail_dq) pairs
                r += tail_dr;
                qq += tail_dq;
                if (qq >= p.tail_pairs) { qq -= p.tail_pairs; ++r; }
            }
        }
        __syncwarp();
        if (lane == 0 && j + D < mine) {
            fence_proxy_async_smem();
            issue(plg, pc, pst);
            next_item(plg, pc);
            if (++pst == D) pst = 0;
        }
        // reduce the item's V row partials across the warp, store them
        float vals[V];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) vals[m * R + r] = acc[m][r];
        const float tot = transpose_reduce<V>(vals, lane);
        if ((lane & (32 / V - 1)) == 0) part[(size_t)it * V + value_of_lane<V>(lane)] = tot;
        // advance: next stage of the ring, next item of this warp
        if (++s == D) { s = 0; parity ^= 1u; }
        next_item(lg, c);
    }
    if (j < mine && lane == 0) {
        // A copy never arrived.  Give the stages already in flight the same
        // bounded time to land in this CTA's shared memory before leaving.
        for (int jj = j + 1; jj < min(mine, j + D); ++jj)
            mbar_wait_bounded(bars + 8u * (uint32_t)(jj % D), (uint32_t)(jj / D) & 1u, p.fault,
                              kFaultBulkWaitTimeout);
    }
    __syncthreads();

    // every row of this CTA: add its partials in chunk order, write the output
    const int nrows = (g1 - g0) * R;
    for (int t = threadIdx.x; t < nrows; t += blockDim.x) {
        const int lg = t / R, r = t - lg * R;
        const int64_t row = (int64_t)(g0 + lg) * R + r;
        if (row >= p.N) continue;
        float sum[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            float a = 0.f;
            for (int c = 0; c < nitems; ++c) a += part[(size_t)(lg * nitems + c) * V + m * R + r];
            sum[m] = a;
        }
        float v = sum[0];
        if constexpr (NMAT == 2) v = gelu_tanh(sum[0]) * sum[1];
        if (p.y_bf16) store_out<__nv_bfloat16>(p.y, row, v);
        else store_out<float>(p.y, row, v);
    }
}

// Host-side launch of one instantiation, as a programmatic dependent of the
// preceding kernel on the stream (the kernel waits for it before reading x).
template <int FMT, int NMAT, int R>
cudaError_t launch_stream_instance(const StreamParams& p, int ctas, int warps, size_t smem,
                                   cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)(warps * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, qmv_stream_kernel<FMT, NMAT, R>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int FMT, int NMAT, int R>
cudaError_t prepare_stream_instance(size_t smem) {
    return cudaFuncSetAttribute(qmv_stream_kernel<FMT, NMAT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
}

}  // namespace qbw
