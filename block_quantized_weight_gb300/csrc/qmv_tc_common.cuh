// qmv_tc_common.cuh -- the operand layout, code decode, activation table and
// read-back pieces of the tensor-core Q4_0 / Q4_K matrix-vector products,
// shared by the one-call kernels (qmv_tc.cu) and the chained form
// (qmv_chain.cu).
#pragma once

#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"
#include "tc_common.cuh"

namespace qbw {
namespace qtc {

using namespace tc;

constexpr int kTileRows = 128;
constexpr int kGroupK = 256;
constexpr int kGroupWords = 18;                  // 144 raw bytes per row per group, as 8-byte TMA words
constexpr int kSets = 3;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp0 = 13;                    // set s's issuer: warp 13 + s
constexpr int kThreads = 16 * 32;
constexpr int kStages = 6;                       // a multiple of kSets: stage s always serves set s % 3
constexpr int kN = 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = kGroupK / 2;         // 128 TMEM columns of A per set
constexpr uint32_t kDCol = kSets * kACols;       // set s's two D buffers at columns 384 + 32 s (+ 16)
constexpr uint32_t kRawStageBytes = kTileRows * 144;
constexpr uint32_t kBBytes = kN * kGroupK * 2;   // 8 KB: 4 swizzle atoms of 16 rows x 128 B
constexpr int kMaxLocalTiles = 8;
constexpr uint32_t kBf16Minus136 = 0xC308C308u;
constexpr uint32_t kBf16Minus128 = 0xC300C300u;

constexpr uint32_t kOffB = kStages * kRawStageBytes;                          // 1024-aligned
// 8-bit form with fp32 activations: a second B per set, the third pieces
constexpr uint32_t kOffB2 = kOffB + kSets * kBBytes;
constexpr uint32_t kOffPart = kOffB2 + kSets * kBBytes;
// The mixed-bit forms (kFmtMix4, kFmtMix2; bf16 activations only): a unit's
// codes, 128 (int4) or 64 (int2) bytes per row, land at the start of its stage
// with the 128-byte swizzle (16-byte chunk j of row r at 16 (j ^ (r mod 8)))
// or the 64-byte swizzle (at 16 (j ^ (r / 2 mod 4))); its 8 fp16 scales and,
// for int4, 8 fp16 biases per row (16 bytes each, row after row) land in the
// B2 region, which only the fp32 form's third pieces use otherwise: stage s's
// scales at kOffB2 + s kMixScaleBytes, its biases 2 KB further on.
constexpr uint32_t kMixCodeBytes = kTileRows * 128;
constexpr uint32_t kMixScaleBytes = 2 * kTileRows * 16;
constexpr uint32_t kMixStageBytes = kMixCodeBytes + kMixScaleBytes;
constexpr uint32_t kMix2StageBytes = kTileRows * 64 + kTileRows * 16;
// int8: a unit's 256 code bytes per row take two ring stages; each holds 128
// of them (128-byte swizzle) and, after them, the unit's 8 scales per row
constexpr uint32_t kMix8StageBytes = kMixCodeBytes + kTileRows * 16;
static_assert(kMix8StageBytes <= kRawStageBytes && kStages % 2 == 0 && (kStages / 2) % kSets == 0,
              "the int8 form's half-units fill the ring two stages per unit, each set on its own pair");
static_assert(kMixCodeBytes <= kRawStageBytes && kStages * kMixScaleBytes <= kSets * kBBytes,
              "the mixed-bit form's stages fit the raw ring and the B2 region");
static_assert(kRawStageBytes % 1024 == 0 && kOffB2 % 1024 == 0, "swizzled copies want 1024-byte aligned stages");
constexpr uint32_t kOffBar = kOffPart + kSets * kMaxLocalTiles * 2 * kTileRows * 4;
constexpr int kBars = 2 * kStages + 4 * kSets + 1;
constexpr uint32_t kOffSlot = kOffBar + 8 * kBars;
// a word set to 1 by the table build when some group of the table is flagged
constexpr uint32_t kOffXflag = kOffSlot + 8;
// 8-bit form: the activations of up to kXtGroups K-groups, built once per CTA:
// per group 32 chunks of 8 elements as {piece 0, piece 1} (16 bytes each),
// with fp32 activations a third piece (8 bytes each), and per group the 8
// blocks' read-back factors c_j (fp32)
constexpr int kXtGroups = 48;
constexpr uint32_t kOffXt = (kOffSlot + 16 + 15) & ~15u;
constexpr uint32_t kOffXt2 = kOffXt + kXtGroups * 32 * 16;
constexpr uint32_t kOffXc = kOffXt2 + kXtGroups * 32 * 8;
constexpr uint32_t kOffXs = kOffXc + kXtGroups * 8 * 4;        // Q4_K: per block sum of x (fp32)
// Per block a_j = Wmax (1 + eps) sum |x_k - pieces_k| over its elements
// (unscaled, fp32; Wmax = 8 for Q4_0 codes, 15 for Q4_K's): the read-back's
// bound on what the pieces miss, per unit of the block scale (see
// unit_check_term); valid for a group whose flag is set.  The flag (some
// element not carried exactly by its pieces) is the sign bit of the group's
// first read-back factor c_0 at kOffXc, which is otherwise positive.
constexpr uint32_t kOffXr = kOffXs + kXtGroups * 8 * 4;
// Per dequantizing thread (a row of a set): the error-check term of the
// segment being accumulated, per matrix (fp32), and the bits of its flagged
// segments (see the read-back of the 8-bit form); zero at the start.
constexpr uint32_t kOffQ = kOffXr + kXtGroups * 8 * 4;
constexpr uint32_t kOffFix = kOffQ + kProducerWarp * 32 * 2 * 4;
constexpr uint32_t kSmemBytes = kOffFix + kProducerWarp * 32 * 4;
// The pieces' error over a segment of a row's units is accepted while it is
// at most kPieceEps of a lower bound of the row's sum |w x| over the segment;
// otherwise the segment's residuals are added exactly.  Elements whose
// residual is not formed (the fp32 form's, within 2^-12) add at most 2^-12
// more.
constexpr float kPieceEps = 0x1p-11f;
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");

static_assert(kStages % kSets == 0, "stage s must serve set s % 3");
static_assert(kOffB % 1024 == 0, "B operand needs 1024-byte alignment");

struct QtcParams {
    CUtensorMap tmap_w[2];   // Q4_0 rows as 8-byte words, box (18, 128); [1]: the up matrix of gate+up
    // the launch that follows on the stream when a chain runs as separate
    // launches (next_units = 0: none): its weights' tensor maps and unit
    // split, so that each CTA's producer can prefetch into L2 the first units
    // the same CTA index loads there
    CUtensorMap next_tmap[2];
    int32_t next_units, next_groups, next_nmat, next_ctas;
    // the mixed-bit forms: tmap_w[0] views the codes as 8-byte words; with
    // groups of 32 (mgshift = 5) tmap_w[1] the fp16 scales and tmap_bi the fp16
    // biases as 8-byte words, box (2, 128).  msc and mbi are the scales and
    // biases ([N][K >> mgshift], one per 2^mgshift weights of a row), which
    // the threads read themselves for larger groups (and for the read-back
    // correction)
    CUtensorMap tmap_bi;
    const uint16_t* msc;
    const uint16_t* mbi;
    int32_t mgshift;
    const void* x;
    void* y;
    unsigned int* fault;
    int32_t N, K;
    int32_t tiles, groups, units;     // units = tiles x groups x matrices
    int32_t x_bf16, y_bf16;
    const uint8_t* w[2];              // the raw weights (w[1]: the up matrix), for the read-back correction
    int64_t row_bytes;
};

__device__ __forceinline__ uint32_t full_bar(uint32_t b0, int s) { return b0 + 8u * (uint32_t)s; }
__device__ __forceinline__ uint32_t empty_bar(uint32_t b0, int s) { return b0 + 8u * (uint32_t)(kStages + s); }
// afull(a, h): half h (K 128h .. 128h + 127) of set a's A and B operands is
// written; aempty(a, h): the MMAs reading that half have completed.
__device__ __forceinline__ uint32_t afull_bar(uint32_t b0, int a, int h) {
    return b0 + 8u * (uint32_t)(2 * kStages + 2 * a + h);
}
__device__ __forceinline__ uint32_t aempty_bar(uint32_t b0, int a, int h) {
    return b0 + 8u * (uint32_t)(2 * kStages + 2 * kSets + 2 * a + h);
}
__device__ __forceinline__ uint32_t done_bar(uint32_t b0) { return b0 + 8u * (uint32_t)(2 * kStages + 4 * kSets); }

// per-set partial rows in shared memory: [set][local tile][matrix][row]
__device__ __forceinline__ int part_at(int set, int lt, int m, int row) {
    return ((set * kMaxLocalTiles + lt) * 2 + m) * kTileRows + row;
}

__device__ __forceinline__ int unit_begin(int c, int units, int ctas) {
    return (int)(((int64_t)units * c) / ctas);
}

// the CTA whose unit range holds unit u
__device__ __forceinline__ int owner_of(int u, int units, int ctas) {
    int c = (int)(((int64_t)u * ctas) / units);
    while (c + 1 < ctas && unit_begin(c + 1, units, ctas) <= u) ++c;
    while (c > 0 && unit_begin(c, units, ctas) > u) --c;
    return c;
}

// One Q4_0 block of the row's group (qs[0] at byte OFF of the words v[]) ->
// 16 bf16x2 columns of exact codes c - 8 in K order: column t holds elements
// 2t and 2t + 1 (t < 8) or 16 + 2(t - 8) and 17 + 2(t - 8).
template <int OFF>
__device__ __forceinline__ void codes_block(const uint32_t (&v)[36], uint32_t* col) {
    const uint32_t m136 = kBf16Minus136;
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        const int byte = OFF + j;
        uint32_t lo, hi;
        if ((byte & 3) == 0) nibble_pairs<0>(v[byte >> 2], lo, hi);
        else nibble_pairs<2>(v[byte >> 2], lo, hi);
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[j >> 1]) : "r"(lo), "r"(m136));
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[8 + (j >> 1)]) : "r"(hi), "r"(m136));
    }
}

// Q4_0: block pair P (blocks 2P, 2P + 1) of the group -> 32 columns of exact
// c - 8.  Q4_K: 64-weight chunk P of the super-block -> 32 columns of exact
// codes c (0..15): its 32 nibble bytes (words 4 + 8P .. 11 + 8P) hold weights
// 64P + l in the low nibbles and 64P + 32 + l in the high nibbles, so the
// byte pair (l, l + 1) gives columns 16 * 0 + l / 2 (low) and 16 + l / 2
// (high) of the chunk, in K order.
template <int FMT, int P>
__device__ __forceinline__ void codes_pair(const uint32_t (&v)[36], uint32_t (&col)[32]) {
    if constexpr (FMT == kFmtQ4) {
        codes_block<36 * P + 2>(v, col);
        codes_block<36 * P + 20>(v, col + 16);
    } else {
        const uint32_t m128 = kBf16Minus128;
#pragma unroll
        for (int wd = 0; wd < 8; ++wd) {
            const uint32_t w = v[4 + 8 * P + wd];
            uint32_t lo, hi;
            nibble_pairs<0>(w, lo, hi);                     // bytes 4wd, 4wd + 1
            asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[2 * wd]) : "r"(lo), "r"(m128));
            asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[16 + 2 * wd]) : "r"(hi), "r"(m128));
            nibble_pairs<2>(w, lo, hi);                     // bytes 4wd + 2, 4wd + 3
            asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[2 * wd + 1]) : "r"(lo), "r"(m128));
            asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(col[16 + 2 * wd + 1]) : "r"(hi), "r"(m128));
        }
    }
}

// 8-bit form of block pair P (blocks 2P, 2P + 1) of a Q4_0 group -> 32 TMEM
// columns of e4m3 bytes, 4 per column in K order.  An e4m3 byte b = 0..15 is
// exactly b * 2^-9 (the subnormals and the first binade share one spacing), so
// code c - 8 = (c & 7) - 8 [c < 8] splits into two exact 8-bit operands that
// are both 0 where c = 8: block j's K-step 2j holds c & 7 and K-step 2j + 1
// holds 8 [bit 3 of c clear] (the byte 0x08), against B columns of +x and -x.
// Each K-step is 8 columns: the low nibbles of qs[0..15] (elements 0..15),
// then their high nibbles (elements 16..31).  Block 2P's qs start at byte
// 36P + 2 of the group row (two bytes into a word), block 2P + 1's at word
// 9P + 5.
template <int P>
__device__ __forceinline__ void codes_pair_e4m3(const uint32_t (&v)[36], uint32_t (&col)[32]) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t w = __funnelshift_r(v[9 * P + t], v[9 * P + t + 1], 16);
        const uint32_t h = __funnelshift_r(v[9 * P + t], v[9 * P + t + 1], 20);
        col[t] = w & 0x07070707u;
        col[4 + t] = h & 0x07070707u;
        col[8 + t] = ~w & 0x08080808u;
        col[12 + t] = ~h & 0x08080808u;
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t w = v[9 * P + 5 + t];
        const uint32_t h = w >> 4;
        col[16 + t] = w & 0x07070707u;
        col[20 + t] = h & 0x07070707u;
        col[24 + t] = ~w & 0x08080808u;
        col[28 + t] = ~h & 0x08080808u;
    }
}

// 8-bit form of Q4_K: half H of a super-block (sub-blocks 4H .. 4H + 3) -> 32
// TMEM columns of e4m3 codes 0..15 (exact, b * 2^-9), one K-step of 8
// columns per sub-block.  Sub-block j is the low (j even) or high (j odd)
// nibbles of 64-weight chunk j / 2, whose 32 bytes are words 4 + 8 (j / 2) ..
// 11 + 8 (j / 2) of the row: byte l holds weight l of the sub-block.
template <int H>
__device__ __forceinline__ void codes_q4k_e4m3(const uint32_t (&v)[36], uint32_t (&col)[32]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int j = 4 * H + s;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = v[4 + 8 * (j >> 1) + t];
            col[8 * s + t] = ((j & 1) ? (w >> 4) : w) & 0x0F0F0F0Fu;
        }
    }
}

// int4-affine mixed-bit form: half H of a unit (groups 4H .. 4H + 3 of 32
// weights, code words 16H .. 16H + 15 of the row's 32) -> 32 TMEM columns of
// e4m3 codes 0..15 (exact, b 2^-9), one K-step of 8 columns per group.  Word
// i of a group holds its weights 8i .. 8i + 7, nibble e = weight 8i + e; the
// even nibbles go to column 2i of the K-step and the odd ones to column 2i +
// 1, so K positions 8i .. 8i + 7 hold weights 8i + 0, 2, 4, 6, 1, 3, 5, 7
// (perm_mix4 puts the activation pieces of B in the same order).
template <int H>
__device__ __forceinline__ void codes_mix4_e4m3(const uint32_t (&v)[36], uint32_t (&col)[32]) {
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const uint32_t w = v[16 * H + t];
        col[2 * t] = w & 0x0F0F0F0Fu;
        col[2 * t + 1] = (w >> 4) & 0x0F0F0F0Fu;
    }
}

// int2-symmetric mixed-bit form: half H of a unit (groups 4H .. 4H + 3, code
// words 8H .. 8H + 7 of the row's 16; a word holds 16 weights, field e in bits
// 2e, 2e + 1) -> 32 TMEM columns of e4m3 values q 2^-9 (exact), one K-step of
// 8 columns per group.  The fields of a 4-weight column are picked as the
// nibbles of a byte-permute selector into a table of the four e4m3 bytes 0,
// +1, -2, -1 (the two's-complement values 0, 1, -2, -1): w masked with
// 0x33333333 holds fields 0, 2, 4, 6 in its low and 8, 10, 12, 14 in its high
// 16 bits, w >> 2 so masked fields 1, 3, 5, 7 and 9, 11, 13, 15 (the permute
// reads the low 16 bits of its selector).  So K positions 8i .. 8i + 7 of a
// group hold its weights 8i + 0, 2, 4, 6, 1, 3, 5, 7, as in the int4 form.
template <int H>
__device__ __forceinline__ void codes_mix2_e4m3(const uint32_t (&v)[36], uint32_t (&col)[32]) {
    constexpr uint32_t kTable = 0x81820100u;     // byte f: e4m3 of the field's value f - 4 (f >> 1)
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t w = v[8 * H + t];
        const uint32_t e = w & 0x33333333u, o = (w >> 2) & 0x33333333u;
        const uint32_t sel[4] = {e, o, e >> 16, o >> 16};
#pragma unroll
        for (int i = 0; i < 4; ++i) asm("prmt.b32 %0, %1, 0, %2;" : "=r"(col[4 * t + i]) : "r"(kTable), "r"(sel[i]));
    }
}

// int8 mixed-bit form: block pair P (blocks 2P, 2P + 1) of the half-unit
// whose 32 code words are v[0..31] (a block's 32 bytes are words 8b .. 8b +
// 7, byte = element) -> 32 TMEM columns, as the two-operand Q4_0 form: block
// b's first K-step (8 columns) holds l = q & 15 (e4m3 bytes l 2^-9, exact)
// and its second holds h = q >> 4 (-8 .. 7) as a signed e4m3 byte h 2^-9
// (exact), against B columns of x and 16 x, so q = l + 16 h.  The signed byte
// is sign | magnitude: with m the byte's sign replicated (a byte permute in
// sign mode), magnitude = (n ^ (m & 15)) + (m & 1) for the high nibble n, and
// the sign bit m & 0x80 joins it in one multiply-add.
template <int P>
__device__ __forceinline__ void codes_mix8_e4m3(const uint32_t (&v)[36], uint32_t (&col)[32]) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t w = v[16 * P + 8 * b + t];
            uint32_t m;
            asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"(w));
            const uint32_t n = (w >> 4) & 0x0F0F0F0Fu;
            col[16 * b + t] = w & 0x0F0F0F0Fu;
            col[16 * b + 8 + t] = (m & 0x01010101u) * 0x81u + (n ^ (m & 0x0F0F0F0Fu));
        }
    }
}

// Eight e4m3 activation pieces times 16, exactly (the int8 form's second
// K-step): through fp16, where the product is exact and the result, below 2^8,
// is representable in e4m3 again.
__device__ __forceinline__ uint2 times16_e4m3(uint2 b) {
    const uint32_t w[2] = {b.x, b.y};
    uint32_t r[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h0, h1;
        asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h0) : "r"(w[i] & 0xFFFFu));
        asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h1) : "r"(w[i] >> 16));
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h0) : "r"(0x4C004C00u));     // x 16
        asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h1) : "r"(0x4C004C00u));
        unsigned short e0, e1;
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e0) : "r"(h0));
        asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e1) : "r"(h1));
        r[i] = (uint32_t)e0 | ((uint32_t)e1 << 16);
    }
    return make_uint2(r[0], r[1]);
}

// The eight bytes of an activation chunk's piece (element order) in the order
// codes_mix4_e4m3 and codes_mix2_e4m3 give a chunk's weights: the even
// elements, then the odd.
__device__ __forceinline__ uint2 perm_mix4(uint2 b) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(lo) : "r"(b.x), "r"(b.y));
    asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(hi) : "r"(b.x), "r"(b.y));
    return make_uint2(lo, hi);
}

// fp16 scales of blocks 2P (low half) and 2P + 1 (high half) of the group:
// block 2P's in the low half of word 9P, block 2P + 1's in the high half of
// word 9P + 4.
__device__ __forceinline__ uint32_t scale_pair(const uint32_t (&v)[36], int P) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, 0x7610;" : "=r"(r) : "r"(v[9 * P]), "r"(v[9 * P + 4]));
    return r;
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t h) {
    float2 f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f.x), "=f"(f.y)
        : "r"(h));
    return f;
}

// Q4_K: the sub-block sums of one unit, r0 = sum_j d sc_j (D[2j] + D[2j + 1])
// - dmin m_j sx_j, j = 0..7 in order: dd[] holds the super-block's first 16
// bytes (fp16 d and dmin, then the 12 six-bit scale bytes), sx the lane's
// sub-block sum of x (lanes 4j .. 4j + 3 hold sub-block j's).
__device__ __forceinline__ float unit_dot_q4k(const uint32_t (&dv)[16], const uint32_t (&dd)[4], float sx) {
    const float2 dm = half2_to_float2(dd[0]);
    const uint32_t s03 = dd[1], s47 = dd[2], s8b = dd[3];       // scale bytes 0..3, 4..7, 8..11
    float r = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t sc, m;
        if (j < 4) {
            sc = (s03 >> (8 * j)) & 63u;
            m = (s47 >> (8 * j)) & 63u;
        } else {
            const uint32_t lo = (s8b >> (8 * (j - 4))) & 0xFFu;
            sc = (lo & 15u) | (((s03 >> (8 * (j - 4) + 6)) & 3u) << 4);
            m = (lo >> 4) | (((s47 >> (8 * (j - 4) + 6)) & 3u) << 4);
        }
        const float sxj = __shfl_sync(0xffffffffu, sx, 4 * j);
        r = fmaf(dm.x * (float)sc, __uint_as_float(dv[2 * j]) + __uint_as_float(dv[2 * j + 1]), r);
        r = fmaf(-dm.y * (float)m, sxj, r);
    }
    return r;
}

// One token (NTOK = 1): r0 = sum_j d_j (D[2j] + D[2j + 1]), the x_hi and x_lo
// columns of block j.  Two tokens: r0 = sum_j d_j D[2j], r1 = sum_j d_j
// D[2j + 1].  j = 0..7 in order.
template <int NTOK>
__device__ __forceinline__ void unit_dot(const uint32_t (&dv)[16], const uint32_t (&dd)[4], float& r0, float& r1) {
    r0 = 0.f;
    r1 = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 d = half2_to_float2(dd[p]);
        if constexpr (NTOK == 1) {
            r0 = fmaf(d.x, __uint_as_float(dv[4 * p]) + __uint_as_float(dv[4 * p + 1]), r0);
            r0 = fmaf(d.y, __uint_as_float(dv[4 * p + 2]) + __uint_as_float(dv[4 * p + 3]), r0);
        } else {
            r0 = fmaf(d.x, __uint_as_float(dv[4 * p]), r0);
            r1 = fmaf(d.x, __uint_as_float(dv[4 * p + 1]), r1);
            r0 = fmaf(d.y, __uint_as_float(dv[4 * p + 2]), r0);
            r1 = fmaf(d.y, __uint_as_float(dv[4 * p + 3]), r1);
        }
    }
}

// 8-bit form, one token: r0 = sum_j (d_j c_j) (D[2j] + D[2j + 1] / 16), j =
// 0..7 in order, where c_j = 2^9 / s_j undoes the e4m3 code scale 2^-9 and
// block j's activation scale s_j (c[0..7] = c_j), and 1/16 the scale of the
// second pieces.
__device__ __forceinline__ float unit_dot_e4m3(const uint32_t (&dv)[16], const uint32_t (&dd)[4], const float (&c)[8]) {
    float r = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 d = half2_to_float2(dd[p]);
        r = fmaf(d.x * fabsf(c[2 * p]), fmaf(__uint_as_float(dv[4 * p + 1]), 0.0625f, __uint_as_float(dv[4 * p])), r);
        r = fmaf(d.y * c[2 * p + 1], fmaf(__uint_as_float(dv[4 * p + 3]), 0.0625f, __uint_as_float(dv[4 * p + 2])), r);
    }
    return r;
}

// 8-bit form of Q4_K: r0 = sum_j (d sc_j c_j) (D[2j] + D[2j + 1] / 16) - dmin m_j sx_j,
// j = 0..7 in order; dd[] holds the super-block's first 16 bytes (fp16 d and
// dmin, then the 12 six-bit scale bytes), c[j] the read-back factors and sx[j]
// the sub-blocks' activation sums.
__device__ __forceinline__ float unit_dot_q4k_e4m3(const uint32_t (&dv)[16], const uint32_t (&dd)[4],
                                                   const float (&c)[8], const float (&sx)[8]) {
    const float2 dm = half2_to_float2(dd[0]);
    const uint32_t s03 = dd[1], s47 = dd[2], s8b = dd[3];
    float r = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t sc, m;
        if (j < 4) {
            sc = (s03 >> (8 * j)) & 63u;
            m = (s47 >> (8 * j)) & 63u;
        } else {
            const uint32_t lo = (s8b >> (8 * (j - 4))) & 0xFFu;
            sc = (lo & 15u) | (((s03 >> (8 * (j - 4) + 6)) & 3u) << 4);
            m = (lo >> 4) | (((s47 >> (8 * (j - 4) + 6)) & 3u) << 4);
        }
        r = fmaf(dm.x * (float)sc * fabsf(c[j]), fmaf(__uint_as_float(dv[2 * j + 1]), 0.0625f, __uint_as_float(dv[2 * j])), r);
        r = fmaf(-dm.y * (float)m, sx[j], r);
    }
    return r;
}

// A mixed-bit unit's eight block values (scales or biases; block 2p in the low
// half of v[p]) from the row's fp16 array of one value per 2^gshift weights
// (gshift >= 5: groups of 32 or more, a power of two), read from global memory
// (the row's array 16-byte aligned for groups of 32, 8 for 64, 4 for 128):
// block j of unit g takes value (256 g + 32 j) >> gshift.
__device__ __forceinline__ void mix_unit_values(const uint16_t* row, int g, int gshift, uint32_t (&v)[4]) {
    const uint16_t* first = row + ((int64_t)g << 8 >> gshift);
    if (gshift == 5) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(first));
        v[0] = w.x;
        v[1] = w.y;
        v[2] = w.z;
        v[3] = w.w;
    } else if (gshift == 6) {
        // four values, one per block pair
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(first));
        v[0] = __byte_perm(w.x, 0u, 0x1010);
        v[1] = __byte_perm(w.x, 0u, 0x3232);
        v[2] = __byte_perm(w.y, 0u, 0x1010);
        v[3] = __byte_perm(w.y, 0u, 0x3232);
    } else if (gshift == 7) {
        // two values, one per four blocks
        const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(first));
        v[0] = v[1] = __byte_perm(w, 0u, 0x1010);
        v[2] = v[3] = __byte_perm(w, 0u, 0x3232);
    } else {
        // one value for the whole unit
        const uint32_t h = __ldg(first);
        v[0] = v[1] = v[2] = v[3] = h | (h << 16);
    }
}

// 8-bit form of the int4-affine mixed-bit matrices: r0 = sum_j (sc_j c_j)
// (D[2j] + D[2j + 1] / 16) + bi_j sx_j, j = 0..7 in order: the split of w = sc
// c + bi, whose codes the pieces multiply while each bias takes its group's
// exact sum of x.  sc[] and bi[] hold the unit's eight fp16 scales and biases
// (group 2p in the low half of word p), c[j] the read-back factors and sx[j]
// the groups' activation sums.
__device__ __forceinline__ float unit_dot_mix4_e4m3(const uint32_t (&dv)[16], const uint32_t (&sc)[4],
                                                    const uint32_t (&bi)[4], const float (&c)[8], const float (&sx)[8]) {
    float r = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 s = half2_to_float2(sc[p]), b = half2_to_float2(bi[p]);
        r = fmaf(s.x * fabsf(c[2 * p]), fmaf(__uint_as_float(dv[4 * p + 1]), 0.0625f, __uint_as_float(dv[4 * p])), r);
        r = fmaf(b.x, sx[2 * p], r);
        r = fmaf(s.y * c[2 * p + 1], fmaf(__uint_as_float(dv[4 * p + 3]), 0.0625f, __uint_as_float(dv[4 * p + 2])), r);
        r = fmaf(b.y, sx[2 * p + 1], r);
    }
    return r;
}

__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// two fp32 -> e4m3 (round to nearest, saturating), lo in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

__device__ __forceinline__ void sts64(uint32_t addr, uint2 v) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo_to_float(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_to_float(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset, in the B operand (K-major, 128-byte swizzle, 16 rows), of the
// 16-byte chunk holding elements 8c .. 8c + 7 of swizzle atom a, row n.
__device__ __forceinline__ uint32_t b_chunk(int a, int n, int c) {
    return (uint32_t)(a * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

// 8-bit form: eight fp32 values of table slot sl at offset off (the read-back
// factors c_j at kOffXc, Q4_K's sub-block sums at kOffXs)
__device__ __forceinline__ void table_f8(uint32_t sbase, uint32_t off, int sl, float (&c)[8]) {
    const uint4 a = lds128(sbase + off + (uint32_t)sl * 32u), b = lds128(sbase + off + (uint32_t)sl * 32u + 16u);
    c[0] = __uint_as_float(a.x);
    c[1] = __uint_as_float(a.y);
    c[2] = __uint_as_float(a.z);
    c[3] = __uint_as_float(a.w);
    c[4] = __uint_as_float(b.x);
    c[5] = __uint_as_float(b.y);
    c[6] = __uint_as_float(b.z);
    c[7] = __uint_as_float(b.w);
}

// Byte offset, in the B operand, of byte `byte` of swizzle atom a, row n
// (the 8-bit form: 128 K-elements per atom row).
__device__ __forceinline__ uint32_t b_byte(int a, int n, uint32_t byte) {
    return (uint32_t)(a * 2048 + (n >> 3) * 1024 + (n & 7) * 128) + ((((byte >> 4) ^ (uint32_t)(n & 7)) << 4) |
                                                                       (byte & 15u));
}

// Eight bf16 activations (x[2e] in the low half of word e), already scaled by
// the power of two sc, as two e4m3 pieces: p0 keeps the sign, exponent and top
// three mantissa bits (fp32 bits & 0xFFF00000), p1 the remaining four bits
// (bf16 has seven) times 16 (below 2^8 for |x| < 2^8, so within e4m3's 448;
// the read-back divides its column by 16).  Both are exact in e4m3 while the
// element is at least 2^-6 after scaling; below that e4m3's subnormal spacing
// of 2^-9 rounds them.
__device__ __forceinline__ void split_e4m3(uint4 xr, float sc, uint2& p0, uint2& p1) {
    const uint32_t w[4] = {xr.x, xr.y, xr.z, xr.w};
    uint32_t h0[4], h1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16) * sc, hi = __uint_as_float(w[e] & 0xFFFF0000u) * sc;
        const float lo0 = __uint_as_float(__float_as_uint(lo) & 0xFFF00000u);
        const float hi0 = __uint_as_float(__float_as_uint(hi) & 0xFFF00000u);
        h0[e] = e4m3x2(lo0, hi0);
        h1[e] = e4m3x2((lo - lo0) * 16.f, (hi - hi0) * 16.f);
    }
    p0 = make_uint2(h0[0] | (h0[1] << 16), h0[2] | (h0[3] << 16));
    p1 = make_uint2(h1[0] | (h1[1] << 16), h1[2] | (h1[3] << 16));
}

// v rounded to four significant bits (sign, exponent, top three mantissa
// bits; half-way cases away from zero): exact in e4m3 in its normal range
__device__ __forceinline__ float round4(float v) { return __uint_as_float((__float_as_uint(v) + 0x00080000u) & 0xFFF00000u); }

// Eight fp32 activations (xa, xb in element order), already scaled by the
// power of two sc, as three e4m3 pieces: p0 = round4(x), p1 = 16 round4(x -
// p0), p2 = e4m3(16 (x - p0 - round4(x - p0))); p1 and p2 share the second
// column, which the read-back divides by 16.  |x - p0| <= 2^-4 |x| and the
// remainder after the second piece is at most 2^-8 |x| (each round4 halves an
// ulp of four bits), so the pieces carry x to 2^-12 relative while the third
// stays in e4m3's normal range (the element at least 2^-2 after scaling).
__device__ __forceinline__ void split3_e4m3(uint4 xa, uint4 xb, float sc, uint2& p0, uint2& p1, uint2& p2) {
    const uint32_t w[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    uint32_t h0[4], h1[4], h2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float a = __uint_as_float(w[2 * e]) * sc, b = __uint_as_float(w[2 * e + 1]) * sc;
        const float a0 = round4(a), b0 = round4(b);
        const float ar = a - a0, br = b - b0;
        const float a1 = round4(ar), b1 = round4(br);
        h0[e] = e4m3x2(a0, b0);
        h1[e] = e4m3x2(a1 * 16.f, b1 * 16.f);
        h2[e] = e4m3x2((ar - a1) * 16.f, (br - b1) * 16.f);
    }
    p0 = make_uint2(h0[0] | (h0[1] << 16), h0[2] | (h0[3] << 16));
    p1 = make_uint2(h1[0] | (h1[1] << 16), h1[2] | (h1[3] << 16));
    p2 = make_uint2(h2[0] | (h2[1] << 16), h2[2] | (h2[3] << 16));
}

__device__ __forceinline__ uint32_t umin16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// two e4m3 bytes (the first element in the low byte) -> two floats
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t b2) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(b2));
    return half2_to_float2(h);
}

// What the e4m3 pieces of one scaled activation v = x s_j leave out: v minus
// the sum of the pieces' values, formed exactly as split_e4m3 (XP = 2) or
// split3_e4m3 (XP = 3) forms the pieces.  Every step is exact in fp32 for bf16
// x; for fp32 x it is within fp32 rounding of the exact residual.
template <int XP>
__device__ __forceinline__ float piece_residual(float v) {
    if constexpr (XP == 2) {
        const float p0 = __uint_as_float(__float_as_uint(v) & 0xFFF00000u);
        const float2 d = e4m3x2_to_float2(e4m3x2(p0, (v - p0) * 16.f));
        return (v - d.x) - d.y * 0.0625f;
    } else {
        const float a0 = round4(v), ar = v - a0, a1 = round4(ar);
        const float2 d01 = e4m3x2_to_float2(e4m3x2(a0, a1 * 16.f));
        const float d2 = e4m3x2_to_float2(e4m3x2((ar - a1) * 16.f, 0.f)).x;
        return ((v - d01.x) - d01.y * 0.0625f) - d2 * 0.0625f;
    }
}

// An element whose scaled exponent e' = E + es - 254 (E its biased fp32
// exponent) is at least kExactExp is carried to 2^-12 relative or better: two
// pieces carry bf16 exactly down to e' = -6 (e4m3's subnormal spacing 2^-9
// reaches the last bit of p0 and of 16 p1 there), and three pieces keep fp32
// to 2^-12 while the third stays in e4m3's normal range (e' >= -2).  Only the
// others need their residual formed.
template <int XP>
constexpr int kExactExp = XP == 2 ? -6 : -2;

// 8-bit form: the activation table of cnt K-groups, group xg0 + sl (mod G) in
// slot sl, from bf16 (XP = 2) or fp32 (XP = 3) x, built by warps w = 0 .. nwarps - 1 of the calling
// group (every lane of each).  Each chunk of 8 elements is scaled by its
// block's s_j = 2^(es - 127), which takes the block's largest |x| into
// [2^7, 2^8) (e4m3 reaches 448); es = 261 - E for the biased exponent E of
// that maximum, kept where s_j and c_j = 2^9 / s_j are normal fp32.
// kCoherent: x may have been written earlier in the same launch by other CTAs
// (loads through L2 only).
template <bool kCoherent>
__device__ __forceinline__ uint4 ld_x16(const void* p) {
    uint4 v;
    if constexpr (kCoherent)
        asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p)
                     : "memory");
    else
        v = __ldg(reinterpret_cast<const uint4*>(p));
    return v;
}

// chunk c of the table (8 elements): bf16 (XP = 2, one 16-byte load) or fp32
// (XP = 3, two)
template <bool kCoherent, int XP>
__device__ __forceinline__ void load_x_chunk(const void* x, int xg0, int G, int c, uint4& xa, uint4& xb) {
    int g = xg0 + (c >> 5);
    if (g >= G) g -= G;
    const size_t e = (size_t)g * kGroupK + 8 * (c & 31);
    if constexpr (XP == 2) {
        xa = ld_x16<kCoherent>(static_cast<const uint16_t*>(x) + e);
    } else {
        xa = ld_x16<kCoherent>(static_cast<const float*>(x) + e);
        xb = ld_x16<kCoherent>(static_cast<const float*>(x) + e + 4);
    }
}

// kLow: the int8 form's table, whose second K-step multiplies the pieces by
// 16: each block's largest |x| goes to [2^3, 2^4) instead of [2^7, 2^8), so
// that 16 times a piece stays below 2^8 (e4m3 reaches 448), and the bound on
// what the pieces miss takes Wmax = 128 (|q| <= 128) per unit of the scale.
template <int XP, bool kSums, bool kLow = false>
__device__ __forceinline__ void table_chunk(uint32_t sbase, int c, int lane, uint4 xa, uint4 xb) {
    if constexpr (kSums) {
        // the block's sum of x (Q4_K's min term): 8 elements per lane, 4 lanes
        float f[8];
        if constexpr (XP == 2) {
            const uint32_t w4[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = __uint_as_float(w4[e] << 16);
                f[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
            }
        } else {
            const uint32_t w8[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(w8[e]);
        }
        float sx = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
        sx += __shfl_xor_sync(0xffffffffu, sx, 1);
        sx += __shfl_xor_sync(0xffffffffu, sx, 2);
        if ((lane & 3) == 0)
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kOffXs + (uint32_t)(c >> 2) * 4u), "f"(sx) : "memory");
    }
    // the block's largest |x|, as bits: bf16 exponent at bit 7, fp32 at bit 23
    uint32_t mx;
    if constexpr (XP == 2) {
        const uint32_t m2 = umax16x2(umax16x2(xa.x & 0x7FFF7FFFu, xa.y & 0x7FFF7FFFu),
                                     umax16x2(xa.z & 0x7FFF7FFFu, xa.w & 0x7FFF7FFFu));
        mx = max(m2 & 0xFFFFu, m2 >> 16) >> 7;
    } else {
        const uint32_t m = max(max(max(xa.x & 0x7FFFFFFFu, xa.y & 0x7FFFFFFFu), max(xa.z & 0x7FFFFFFFu, xa.w & 0x7FFFFFFFu)),
                               max(max(xb.x & 0x7FFFFFFFu, xb.y & 0x7FFFFFFFu), max(xb.z & 0x7FFFFFFFu, xb.w & 0x7FFFFFFFu)));
        mx = m >> 23;
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int es = min(max((kLow ? 257 : 261) - (int)mx, 9), 253);
    const float sc = __uint_as_float((uint32_t)es << 23);
    uint2 q0, q1, q2;
    if constexpr (XP == 2) {
        split_e4m3(xa, sc, q0, q1);
    } else {
        split3_e4m3(xa, xb, sc, q0, q1, q2);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(sbase + kOffXt2 + (uint32_t)c * 8u), "r"(q2.x),
                     "r"(q2.y)
                     : "memory");
    }
    sts128(sbase + kOffXt + (uint32_t)c * 16u, make_uint4(q0.x, q0.y, q1.x, q1.y));
    if ((lane & 3) == 0)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sbase + kOffXc + (uint32_t)(c >> 2) * 4u),
                     "r"((uint32_t)(263 - es) << 23)
                     : "memory");
    // The elements the pieces carry with a relative error above 2^-11: their
    // residuals make the correction exact (the warp's 32 chunks are one
    // group, so the group's list is compacted with a warp prefix sum).
    // Quick test first: the smallest nonzero |x| of the chunk (|x| - 1 as
    // unsigned bits, which sends 0 to the top) against the exponent bound te.
    const int te = max(254 + kExactExp<XP> - es, 1);     // candidates have E < te
    bool any;
    if constexpr (XP == 2) {
        const uint32_t t0 = ((xa.x | 0x80008000u) - 0x00010001u) & 0x7FFF7FFFu;
        const uint32_t t1 = ((xa.y | 0x80008000u) - 0x00010001u) & 0x7FFF7FFFu;
        const uint32_t t2 = ((xa.z | 0x80008000u) - 0x00010001u) & 0x7FFF7FFFu;
        const uint32_t t3 = ((xa.w | 0x80008000u) - 0x00010001u) & 0x7FFF7FFFu;
        const uint32_t m2 = umin16x2(umin16x2(t0, t1), umin16x2(t2, t3));
        any = min(m2 & 0xFFFFu, m2 >> 16) < ((uint32_t)te << 7);
    } else {
        const uint32_t w8[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        uint32_t m = 0xFFFFFFFFu;
#pragma unroll
        for (int e = 0; e < 8; ++e) m = min(m, (w8[e] & 0x7FFFFFFFu) - 1u);
        any = m < ((uint32_t)te << 23);
    }
    const uint32_t slot = (uint32_t)(c >> 5);
    if (!__any_sync(0xffffffffu, any)) return;
    float f[8];
    if constexpr (XP == 2) {
        const uint32_t w4[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w4[e] << 16);
            f[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
        }
    } else {
        const uint32_t w8[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(w8[e]);
    }
    uint32_t cand = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int E = (int)((__float_as_uint(f[e]) >> 23) & 0xFFu);
        if (f[e] != 0.f && E < te) cand |= 1u << e;
    }
    const float inv_sc = __uint_as_float((uint32_t)(254 - es) << 23);
    float rsum = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (cand & (1u << e)) rsum += fabsf(piece_residual<XP>(f[e] * sc));
    rsum *= inv_sc;
    const bool nz = rsum != 0.f;
    // the block's sum: lanes 4j .. 4j + 3 hold block j's 32 elements
    rsum += __shfl_xor_sync(0xffffffffu, rsum, 1);
    rsum += __shfl_xor_sync(0xffffffffu, rsum, 2);
    if ((lane & 3) == 0)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(sbase + kOffXr + (uint32_t)(c >> 2) * 4u),
                     "f"(rsum * (kLow ? 128.f : (kSums ? 15.f : 8.f)) * (1.f + kPieceEps))
                     : "memory");
    // the group's flag: the sign bit of block 0's read-back factor (a
    // positive power of two), stored by lane 0, which holds block 0's es
    if (__any_sync(0xffffffffu, nz) && lane == 0) {
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sbase + kOffXc + slot * 32u),
                     "r"(((uint32_t)(263 - es) << 23) | 0x80000000u)
                     : "memory");
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(sbase + kOffXflag), "r"(1u) : "memory");
    }
}

template <bool kCoherent, int XP, bool kSums = false, bool kLow = false>
__device__ __forceinline__ void build_x_table(uint32_t sbase, const void* x, int xg0, int G, int cnt, int w,
                                              int lane, int nwarps) {
    // a warp's chunks are 32 consecutive ones (block j = lanes 4j .. 4j + 3);
    // up to four per lane are loaded before any is converted, so their L2
    // round trips overlap
    const int nch = cnt * 32;
    const int stride = nwarps * 32;
    for (int c0 = w * 32; c0 < nch; c0 += 4 * stride) {
        uint4 xa[4], xb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (c0 + j * stride < nch) load_x_chunk<kCoherent, XP>(x, xg0, G, c0 + j * stride + lane, xa[j], xb[j]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (c0 + j * stride < nch)
                table_chunk<XP, kSums, kLow>(sbase, c0 + j * stride + lane, lane, xa[j], xb[j]);
    }
}

// The row's weight at element k (0..255) of a unit, exact in fp32, from the
// row's 144 raw bytes b[]: Q4_0 d_j (c - 8) (block j = k / 32, code k % 32 of
// its 16 bytes: low nibbles first); Q4_K d sc_j q, the part the pieces
// multiply (its min term dmin m_j is applied to the exact sum of x); the
// int4-affine form sc_j c (nibble k of the 128 code bytes, lowest first, then
// the eight fp16 scales at byte 128; its bias takes the exact sum of x); the
// int2 form sc_j q (2-bit field k of the 64 code bytes, scales at byte 64);
// the int8 form sc_j q (byte k of the 256 code bytes, scales at byte 256).
template <int FMT>
__device__ __forceinline__ float unit_weight(const uint8_t* b, int k) {
    if constexpr (FMT == kFmtMix8) {
        // byte k of the 256 code bytes (two's complement), scales at byte 256
        const int j = k >> 5;
        return half_bits_to_float((uint32_t)b[256 + 2 * j] | ((uint32_t)b[257 + 2 * j] << 8)) *
               (float)(int)(int8_t)b[k];
    } else if constexpr (FMT == kFmtMix2) {
        // field k of the 64 code bytes (two's complement), scales at byte 64
        const int f = (int)(((uint32_t)b[k >> 2] >> (2 * (k & 3))) & 3u);
        const int j = k >> 5;
        return half_bits_to_float((uint32_t)b[64 + 2 * j] | ((uint32_t)b[65 + 2 * j] << 8)) * (float)(f - 4 * (f >> 1));
    } else if constexpr (FMT == kFmtMix4) {
        const uint32_t code = ((uint32_t)b[k >> 1] >> (4 * (k & 1))) & 15u;
        const int j = k >> 5;
        return half_bits_to_float((uint32_t)b[128 + 2 * j] | ((uint32_t)b[129 + 2 * j] << 8)) * (float)code;
    } else if constexpr (FMT == kFmtQ4) {
        const uint8_t* blk = b + 18 * (k >> 5);
        const int e = k & 31;
        const uint32_t byte = blk[2 + (e & 15)];
        const int code = (int)((e < 16) ? (byte & 15u) : (byte >> 4));
        return half_bits_to_float((uint32_t)blk[0] | ((uint32_t)blk[1] << 8)) * (float)(code - 8);
    } else {
        const int j = k >> 5;
        const uint32_t byte = b[16 + 32 * (k >> 6) + (k & 31)];
        const uint32_t q = (j & 1) ? (byte >> 4) : (byte & 15u);
        const uint32_t sc = j < 4 ? (b[4 + j] & 63u) : ((b[4 + j + 4] & 15u) | ((uint32_t)(b[4 + j - 4] >> 6) << 4));
        return half_bits_to_float((uint32_t)b[0] | ((uint32_t)b[1] << 8)) * (float)sc * (float)q;
    }
}

// 8-bit form, one unit of one row: its term of the read-back's error check.
// With t_j the computed scaled dot of block j (what the read-back adds) and
// R_j the table's sum of |x_k - pieces_k| over block j, E = sum_j Wmax_j R_j
// bounds what the pieces miss (Wmax_j: the block's largest |weight|, 8 |d_j|
// for Q4_0, 15 |d sc_j| for Q4_K), and L = sum_j |t_j| - E is a lower bound
// of the row's sum |w x| over the unit (|t_j| <= sum_k |w_k x_k| + the
// block's error).  The term is q = E (1 + eps) - eps sum_j |t_j|: a segment of
// units whose terms sum to at most 0 has E <= eps L, so its error is at most
// eps of its sum |w x|.  The table holds a_j = (1 + eps) Wmax_j R_j per unit
// of the block scale (|d_j| for Q4_0, |d sc_j| for Q4_K), so q = sum_j
// scale_j (a_j - eps c_j |D_j|) with D_j the block's two columns combined.
template <int FMT>
__device__ __forceinline__ float unit_check_term(const uint32_t (&dv)[16], const uint32_t (&dd)[4], const float (&c)[8],
                                                 const float (&a)[8]) {
    float q = 0.f;
    if constexpr (FMT == kFmtQ4 || FMT == kFmtMix4 || FMT == kFmtMix2 || FMT == kFmtMix8) {
        // dd[p]: the scales of blocks 2p and 2p + 1 as an fp16 pair (Q4_0's d,
        // the mixed-bit forms' sc)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float2 d = half2_to_float2(dd[p]);
            const float D0 = fmaf(__uint_as_float(dv[4 * p + 1]), 0.0625f, __uint_as_float(dv[4 * p]));
            const float D1 = fmaf(__uint_as_float(dv[4 * p + 3]), 0.0625f, __uint_as_float(dv[4 * p + 2]));
            q = fmaf(fabsf(d.x), fmaf(-kPieceEps * fabsf(c[2 * p]), fabsf(D0), a[2 * p]), q);
            q = fmaf(fabsf(d.y), fmaf(-kPieceEps * c[2 * p + 1], fabsf(D1), a[2 * p + 1]), q);
        }
    } else {
        const float dq = fabsf(half2_to_float2(dd[0]).x);
        const uint32_t s03 = dd[1], s8b = dd[3];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t sc;
            if (j < 4) {
                sc = (s03 >> (8 * j)) & 63u;
            } else {
                const uint32_t lo = (s8b >> (8 * (j - 4))) & 0xFFu;
                sc = (lo & 15u) | (((s03 >> (8 * (j - 4) + 6)) & 3u) << 4);
            }
            const float D = fmaf(__uint_as_float(dv[2 * j + 1]), 0.0625f, __uint_as_float(dv[2 * j]));
            q = fmaf(dq * (float)sc, fmaf(-kPieceEps * fabsf(c[j]), fabsf(D), a[j]), q);
        }
    }
    return q;
}

// Whether table slot sl's group has a flag (its read-back factor c_0 < 0).
__device__ __forceinline__ bool group_flagged(uint32_t sbase, int sl) {
    return (lds32(sbase + kOffXc + (uint32_t)sl * 32u) >> 31) != 0u;
}

// The check itself, over a segment of a row's units: the segment needs its
// residuals added exactly when the sum of its units' check terms is above 0,
// i.e. when the pieces may miss more than eps of the segment's sum |w x|.
__device__ __forceinline__ bool segment_needs_correction(float q) { return q > 0.f; }

// The exact sum of w_k r_k over a unit's 256 elements, r_k = x_k minus what
// its pieces carry, formed again from x (group g, elements 256 g ..
// 256 g + 255; block scales from table slot sl) and the row's raw bytes read
// from global memory at wrow (16-byte aligned; the stage holding them has
// long been released): 144 bytes, or for the mixed-bit forms 256 (int8), 128
// (int4) or 64 (int2) code bytes and the unit's eight block scales sc8 (block
// 2p in the low half of word p).  For the segments the read-back check flags;
// slow, and exact up to fp32 rounding.
template <int FMT, int XP, bool kCoherent>
__device__ __noinline__ float unit_correction(const uint8_t* wrow, const void* x, int g, uint32_t sbase, int sl,
                                              uint4 sc8 = make_uint4(0u, 0u, 0u, 0u)) {
    // 16-byte pieces of the row's unit: codes, then (mixed-bit) the scales
    constexpr int kCodeChunks = FMT == kFmtMix8 ? 16 : (FMT == kFmtMix2 ? 4 : (FMT == kFmtMix4 ? 8 : 9));
    constexpr bool kScales = FMT == kFmtMix2 || FMT == kFmtMix4 || FMT == kFmtMix8;
    uint8_t b[FMT == kFmtMix8 ? 272 : 144];
#pragma unroll
    for (int j = 0; j < kCodeChunks; ++j)
        *reinterpret_cast<uint4*>(b + 16 * j) = __ldg(reinterpret_cast<const uint4*>(wrow + 16 * j));
    if constexpr (kScales) *reinterpret_cast<uint4*>(b + 16 * kCodeChunks) = sc8;
    float corr = 0.f;
    for (int k = 0; k < kGroupK; ++k) {
        const uint32_t cb = lds32(sbase + kOffXc + (uint32_t)sl * 32u + (uint32_t)(k >> 5) * 4u);
        const int es = 263 - (int)((cb >> 23) & 0xFFu);
        const float sc = __uint_as_float((uint32_t)es << 23), inv_sc = __uint_as_float((uint32_t)(254 - es) << 23);
        const size_t i = (size_t)g * kGroupK + (size_t)k;
        float xv;
        if constexpr (XP == 2) {
            unsigned short h;
            if constexpr (kCoherent)
                asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(static_cast<const uint16_t*>(x) + i) : "memory");
            else
                h = __ldg(static_cast<const unsigned short*>(x) + i);
            xv = __uint_as_float((uint32_t)h << 16);
        } else {
            if constexpr (kCoherent)
                asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(xv) : "l"(static_cast<const float*>(x) + i) : "memory");
            else
                xv = __ldg(static_cast<const float*>(x) + i);
        }
        const float r = piece_residual<XP>(xv * sc) * inv_sc;
        if (r != 0.f) corr = fmaf(unit_weight<FMT>(b, k), r, corr);
    }
    return corr;
}

}  // namespace qtc
}  // namespace qbw
