// qmv_tc.cu -- the M = 1 (and two-token) Q4_0 matrix-vector product y = W x,
// the fused Q4_0 gate+up, and the Q4_K product, on the fifth-generation tensor
// cores (tcgen05), for K a multiple of 256.  A Q4_K super-block (256 weights,
// 144 bytes) is exactly one unit's row segment; its codes enter A exactly
// (0..15), and the read-back applies d sc_j to each sub-block's dot product
// and subtracts dmin m_j times the sub-block's activation sum (the algebraic
// split of jouleclaw-loader-gguf BENCHMARKS, Q4_K NEON kernel).
//
// Why tensor cores for one token: on CUDA cores every weight costs a code
// extraction, an exact conversion to fp32 and a multiply-add, about 2.1
// instructions, and that instruction stream, not HBM, bounds the CUDA-core
// kernel.  Here a weight costs about 1.6 instructions: two codes become one
// exact bf16x2 pair (byte permute, LOP3 with the exponent of 128, one packed
// add of -136 that leaves c - 8 exactly), and the products and sums run on the
// tensor core.
//
// Exact block scales.  A = the integer codes c - 8 (exact in bf16); the scale
// d of each block is applied after the MMA, in fp32, so no weight is rounded.
// The MMA's N dimension carries one column pair per block instead of one per
// token: for a K-group of 256 (8 blocks), B is 16 columns x 256 K where column
// 2j holds x_hi and column 2j + 1 holds x_lo over block j's 32 elements and
// zeros elsewhere.  x_hi = bf16(x), x_lo = bf16(x - x_hi): their sum is x to
// 2^-17 relative (bf16 activations are exact: x_lo = 0).  So after the 16 MMAs
// of a group, D[row][2j] + D[row][2j + 1] is the block's exact-code dot
// product sum_i (c_i - 8) x_i in fp32, and the row's thread adds
// d_j * (D[2j] + D[2j + 1]) for j = 0..7, in that order.
//
// Work split (stream-K): the units are (128-row tile, K-group, matrix) triples
// in that order (one matrix, or gate then up); CTA c of C takes units
// [c U / C, (c + 1) U / C).  A tile
// that a CTA covers in full is written to y by that CTA.  A tile split between
// CTAs is finished by the CTA that covers its first unit (it reaches the tile
// last, at the end of its range).  Every other CTA on the tile starts its range
// inside it, completes its share early and publishes it then: one 64-bit word
// per row, (value, 1).  The finisher waits for those words (bounded), adds
// them after its own share in CTA order, writes y and marks them consumed
// (tag 0).  Results are therefore bit-reproducible.
//
// Warp roles (16 warps): warps 0..11 are three sets of four dequantizing
// warps; set s takes the CTA's units s, s + 3, ...; warp 4s + q owns rows
// 32q .. 32q + 31 (its TMEM lane quarter) and one eighth of the group's B
// operand (Q4_0: lanes 0..7; Q4_K: lanes 8q .. 8q + 7, while every lane loads
// activations for the sub-block sums).  Warp 12 lane 0 issues the TMA copies of the raw rows
// (128 rows x 144 bytes per unit) into a 6-stage ring.  Warp 13 + s lane 0
// issues set s's MMAs (M = 128, N = 16, K = 16; 16 per unit) into set s's
// accumulator.  Each set's rows read D back one unit later, while the next
// unit's codes are already decoded in registers.
#include <algorithm>
#include <atomic>
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"
#include "tc_common.cuh"

namespace qbw {

// Split-tile scratch, one slot per call in flight: each CTA's published
// share of its first tile, per row (fp32 bits, tag) with tag 1 = published,
// 0 = consumed (all zero at load).
constexpr int kQtcSlots = 16;
constexpr int kQtcMaxCtas = 160;
constexpr int kQtcMaxTiles = 4096;
__device__ unsigned long long g_qtc_share[kQtcSlots][kQtcMaxCtas][2][128];

namespace {

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
constexpr uint32_t kOffPart = kOffB + kSets * kBBytes;
constexpr uint32_t kOffBar = kOffPart + kSets * kMaxLocalTiles * 2 * kTileRows * 4;
constexpr int kBars = 2 * kStages + 4 * kSets + 1;
constexpr uint32_t kOffSlot = kOffBar + 8 * kBars;
// 8-bit form: the activations of up to kXtGroups K-groups, built once per CTA:
// per group 32 chunks of 8 elements as {piece 0, piece 1} (16 bytes each),
// and per group the 8 blocks' read-back factors c_j (fp32)
constexpr int kXtGroups = 64;
constexpr uint32_t kOffXt = (kOffSlot + 16 + 15) & ~15u;
constexpr uint32_t kOffXc = kOffXt + kXtGroups * 32 * 16;
constexpr uint32_t kSmemBytes = kOffXc + kXtGroups * 8 * 4;

static_assert(kStages % kSets == 0, "stage s must serve set s % 3");
static_assert(kOffB % 1024 == 0, "B operand needs 1024-byte alignment");

struct QtcParams {
    CUtensorMap tmap_w[2];   // Q4_0 rows as 8-byte words, box (18, 128); [1]: the up matrix of gate+up
    const void* x;
    void* y;
    unsigned int* fault;
    int32_t N, K;
    int32_t tiles, groups, units;     // units = tiles x groups x matrices
    int32_t slot;
    int32_t x_bf16, y_bf16;
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

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

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

// 8-bit form, one token: r0 = sum_j (d_j c_j) (D[2j] + D[2j + 1]), j = 0..7 in
// order, where c_j = 2^9 / s_j undoes the e4m3 code scale 2^-9 and block j's
// activation scale s_j (c[0..7] = c_j).
__device__ __forceinline__ float unit_dot_e4m3(const uint32_t (&dv)[16], const uint32_t (&dd)[4], const float (&c)[8]) {
    float r = 0.f;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const float2 d = half2_to_float2(dd[p]);
        r = fmaf(d.x * c[2 * p], __uint_as_float(dv[4 * p]) + __uint_as_float(dv[4 * p + 1]), r);
        r = fmaf(d.y * c[2 * p + 1], __uint_as_float(dv[4 * p + 2]) + __uint_as_float(dv[4 * p + 3]), r);
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

// 8-bit form: the read-back factors c_j of the group in table slot sl
__device__ __forceinline__ void table_c(uint32_t sbase, int sl, float (&c)[8]) {
    const uint4 a = lds128(sbase + kOffXc + (uint32_t)sl * 32u), b = lds128(sbase + kOffXc + (uint32_t)sl * 32u + 16u);
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
// the power of two sc, as two e4m3 pieces whose sum is exact: p0 keeps the
// sign, exponent and top three mantissa bits (fp32 bits & 0xFFF00000), p1
// the remaining four bits (bf16 has seven).  Both are exact in e4m3 while the
// element is at least 2^-2 after scaling; below that e4m3's subnormal spacing
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
        h1[e] = e4m3x2(lo - lo0, hi - hi0);
    }
    p0 = make_uint2(h0[0] | (h0[1] << 16), h0[2] | (h0[3] << 16));
    p1 = make_uint2(h1[0] | (h1[1] << 16), h1[2] | (h1[3] << 16));
}

// NMAT = 1: y = W x.  NMAT = 2: out = gelu_tanh(Wg x) * (Wu x); the units of a
// (tile, group) are its gate and up halves, in that order (measured faster
// than all gate groups of a tile before its up groups, by about 1 %).  NTOK = 2 (with
// NMAT = 1 and bf16 activations): Y[m] = W X[m] for two token rows, which take
// the two B columns of each block that x_hi and x_lo take for one token.
// Each row keeps NCH = NMAT * NTOK sums (channels).  F8: the 8-bit form of
// the operands (Q4_0, one token, bf16 activations; see codes_pair_e4m3).
template <int FMT, int NMAT, int NTOK, bool F8>
__device__ __forceinline__ void qmv_tc_body(const QtcParams& p) {
    constexpr int NCH = NMAT * NTOK;
    static_assert(NCH <= 2, "at most two sums per row");
    static_assert(FMT == kFmtQ4 || (NMAT == 1 && NTOK == 1), "Q4_K: one matrix, one token");
    static_assert(!F8 || (FMT == kFmtQ4 && NTOK == 1), "8-bit form: Q4_0, one token");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ctas = (int)gridDim.x, cta = (int)blockIdx.x;
    const int G = p.groups, GU = p.groups * NMAT;    // K-groups, units per tile
    const int u0 = unit_begin(cta, p.units, ctas), u1 = unit_begin(cta + 1, p.units, ctas);
    const int n = u1 - u0;
    const int tile0 = u0 / GU;
    // this CTA starts inside its first tile: it publishes its share of it early
    const bool contrib0 = n > 0 && tile0 * GU < u0;
    __shared__ unsigned int qcount[4];
    if (threadIdx.x < 4) qcount[threadIdx.x] = 0u;
    unsigned long long* share = &g_qtc_share[p.slot][0][0][0];   // [cta][matrix][row]

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    float* part = reinterpret_cast<float*>(smem + kOffPart);      // [set][local tile][matrix][row]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
    bool ok = true;

    // zero B operands (only their fixed activation positions are ever written
    // again) and the per-set partial rows
    for (int i = threadIdx.x; i < (int)(kSets * kBBytes / 16); i += kThreads)
        sts128(sbase + kOffB + 16u * (uint32_t)i, make_uint4(0u, 0u, 0u, 0u));
    for (int i = threadIdx.x; i < kSets * kMaxLocalTiles * 2 * kTileRows; i += kThreads) part[i] = 0.f;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(full_bar(bar0, s), 1);
                mbar_init(empty_bar(bar0, s), 4);
            }
            for (int a = 0; a < kSets; ++a)
                for (int h = 0; h < 2; ++h) {
                    mbar_init(afull_bar(bar0, a, h), 4);
                    mbar_init(aempty_bar(bar0, a, h), 1);
                }
            mbar_init(done_bar(bar0), kSets);
            fence_mbar_init();
        }
        __syncwarp();
        fence_proxy_async_smem();
        asm volatile("bar.arrive 1, %0;" ::"n"(kThreads) : "memory");
        if (lane == 0) {
            prefetch_tmap(&p.tmap_w[0]);
            if (NMAT == 2) prefetch_tmap(&p.tmap_w[1]);
            // weights do not depend on the preceding grid: start streaming now
            for (int i = 0; i < n && ok; ++i) {
                const int s = i % kStages;
                if (i >= kStages)
                    ok = mbar_wait_bounded(empty_bar(bar0, s), (uint32_t)((i / kStages) - 1) & 1u, p.fault,
                                           kFaultBulkWaitTimeout);
                if (!ok) break;
                const int u = u0 + i, ug = u / NMAT, mat = u - ug * NMAT, t = ug / G, g = ug - t * G;
                mbar_arrive_expect_tx(full_bar(bar0, s), kRawStageBytes);
                tma_load_2d(sbase + (uint32_t)s * kRawStageBytes, &p.tmap_w[mat], g * kGroupWords, t * kTileRows,
                            full_bar(bar0, s), policy_evict_first());
            }
        }
    } else {
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "n"(kTmemCols));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
        tc_fence_after();
    }
    // x and y belong to the preceding grid's stream order
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp >= kMmaWarp0) {
        // ---------------- MMA issuer of set s: 16 K-steps per unit into D_s
        const int set = warp - kMmaWarp0;
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            const uint32_t idesc = F8 ? idesc_e4m3(kTileRows, kN) : idesc_bf16(kTileRows, kN);
            const uint32_t a_tmem = tmem + (uint32_t)set * kACols;
            const uint64_t b0 = sw128_desc(sbase + kOffB + (uint32_t)set * kBBytes);
            uint32_t phase = 0;
            for (int i = set; i < n; i += kSets) {
                // the set's k-th unit accumulates into D buffer k % 2
                const uint32_t d_tmem = tmem + kDCol + 32u * (uint32_t)set + 16u * phase;
                // K-steps 0..7 as soon as the first half is written, 8..15 after the second
                ok = mbar_wait_bounded(afull_bar(bar0, set, 0), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t bd = b0 + (uint64_t)((k >> 2) * 128 + (k & 3) * 2);
                    if constexpr (F8) tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, bd, idesc, k > 0 ? 1u : 0u);
                    else tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, bd, idesc, k > 0 ? 1u : 0u);
                }
                tc_commit(aempty_bar(bar0, set, 0));
                ok = mbar_wait_bounded(afull_bar(bar0, set, 1), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 8; k < 16; ++k) {
                    const uint64_t bd = b0 + (uint64_t)((k >> 2) * 128 + (k & 3) * 2);
                    if constexpr (F8) tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, bd, idesc, 1u);
                    else tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, bd, idesc, 1u);
                }
                tc_commit(aempty_bar(bar0, set, 1));
                phase ^= 1u;
            }
            // completes when every MMA issued above has finished
            tc_commit(done_bar(bar0));
        }
    } else if (warp < kProducerWarp) {
        // ---------------- dequantizing warp: set s, lane quarter q
        const int set = warp >> 2, q = warp & 3;
        const uint32_t tmem = *tmem_slot;
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        const uint32_t a_taddr = tmem + lanes + (uint32_t)set * kACols;
        const uint32_t d_taddr = tmem + lanes + kDCol + 32u * (uint32_t)set;   // + 16 (k % 2)
        const uint32_t raw_row = (uint32_t)(32 * q + lane) * 144u;
        const uint32_t bbuf = sbase + kOffB + (uint32_t)set * kBBytes;
        // The lane's 8-element slot xl of the group's activations: Q4_0, lanes
        // 0..7 load slots 8q .. 8q + 7 and write them into B; Q4_K, every lane
        // loads slot `lane` (the sub-block sums need all 256) and the lanes of
        // slots 8q .. 8q + 7 write them.  Slot xl is elements 8 xl .. 8 xl + 7 of
        // the group: swizzle atom xl / 8, block j = xl / 4, B rows 2j (x_hi)
        // and 2j + 1 (x_lo), in K-half xl / 16.
        // (the 8-bit form's B-writing lanes read their slot from the table)
        constexpr bool kAllLanesX = FMT == kFmtQ4K;
        const int xl = kAllLanesX ? lane : 8 * q + lane;
        const bool loads_x = !F8 && (kAllLanesX || lane < 8);
        const bool bwriter = kAllLanesX ? ((lane >> 3) == q) : (lane < 8);
        const int bj = xl >> 2;
        const uint32_t b_hi = bbuf + b_chunk(xl >> 3, 2 * bj, xl & 7);
        const uint32_t b_lo = bbuf + b_chunk(xl >> 3, 2 * bj + 1, xl & 7);
        // 8-bit form: the slot's 8 bytes in K-steps 2j (+x) and 2j + 1 (-x),
        // rows 2j (piece 0) and 2j + 1 (piece 1), atom j / 2
        const uint32_t bo = (uint32_t)((bj & 1) * 64 + 8 * (xl & 3));
        const uint32_t f8_p0 = bbuf + b_byte(bj >> 1, 2 * bj, bo), f8_p1 = bbuf + b_byte(bj >> 1, 2 * bj + 1, bo);
        const uint32_t f8_n0 = bbuf + b_byte(bj >> 1, 2 * bj, bo + 32u);
        const uint32_t f8_n1 = bbuf + b_byte(bj >> 1, 2 * bj + 1, bo + 32u);
        const int bhalf = xl >> 4;
        const int row = 32 * q + lane;
        // 8-bit form: the table of the K-groups g of this CTA's units, group g
        // in slot (g - xg0) mod G.  Each chunk of 8 elements is scaled by its
        // block's s_j = 2^(es - 127), which takes the block's largest |x| into
        // [2^7, 2^8) (e4m3 reaches 448); es = 261 - E for the bf16 biased
        // exponent E of that maximum, kept where s_j and c_j = 2^9 / s_j are
        // normal fp32.  Built by the twelve dequantizing warps; the host
        // launches this form only where the table holds every group needed.
        const int xg0 = (u0 / NMAT) % G;
        if constexpr (F8) {
            const int cnt = n > 0 ? min(G, (u1 - 1) / NMAT - u0 / NMAT + 1) : 0;
            if (cnt > kXtGroups) record_fault(p.fault, kFaultPlan);
            const int nch = min(cnt, kXtGroups) * 32;
            for (int c0 = warp * 32; c0 < nch; c0 += kProducerWarp * 32) {
                const int c = c0 + lane, sl = c >> 5;
                int g = xg0 + sl;
                if (g >= G) g -= G;
                const uint4 xr = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                                      (size_t)g * kGroupK + 8 * (c & 31)));
                const uint32_t m2 = umax16x2(umax16x2(xr.x & 0x7FFF7FFFu, xr.y & 0x7FFF7FFFu),
                                             umax16x2(xr.z & 0x7FFF7FFFu, xr.w & 0x7FFF7FFFu));
                uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const int es = min(max(261 - (int)(mx >> 7), 9), 253);
                uint2 q0, q1;
                split_e4m3(xr, __uint_as_float((uint32_t)es << 23), q0, q1);
                sts128(sbase + kOffXt + (uint32_t)c * 16u, make_uint4(q0.x, q0.y, q1.x, q1.y));
                if ((lane & 3) == 0)
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(sbase + kOffXc + (uint32_t)(c >> 2) * 4u),
                                 "r"((uint32_t)(263 - es) << 23)
                                 : "memory");
            }
            asm volatile("bar.sync 2, %0;" ::"n"(kProducerWarp * 32) : "memory");
        }
        bool counted = !contrib0;
        // after the three sets' shares of the first tile are in part[][0][], the
        // last of a quarter's three warps publishes the quarter's rows
        auto count_in = [&]() {
            __syncwarp();
            unsigned int old = 0;
            if (lane == 0) {
                __threadfence_block();
                old = atomicAdd(&qcount[q], 1u);
            }
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == kSets - 1) {
                __threadfence_block();
#pragma unroll
                for (int m = 0; m < NCH; ++m) {
                    const float v = part[part_at(0, 0, m, row)] + part[part_at(1, 0, m, row)] +
                                    part[part_at(2, 0, m, row)];
                    st_relaxed_u64(share + ((size_t)cta * 2 + m) * kTileRows + row,
                                   (unsigned long long)__float_as_uint(v) | (1ull << 32));
                }
            }
            counted = true;
        };
        // the row's sums of the tile being accumulated, one per matrix
        float acc[NCH];
#pragma unroll
        for (int m = 0; m < NCH; ++m) acc[m] = 0.f;
        int acc_tile = -1, pend_tile = -1, pend_mat = 0;
        auto add_unit = [&](float r0, float r1) {
            if (pend_tile != acc_tile) {
                if (acc_tile >= 0)
#pragma unroll
                    for (int m = 0; m < NCH; ++m) part[part_at(set, acc_tile - tile0, m, row)] = acc[m];
#pragma unroll
                for (int m = 0; m < NCH; ++m) acc[m] = 0.f;
                acc_tile = pend_tile;
                if (!counted && pend_tile > tile0) count_in();
            }
            if constexpr (NTOK == 2) {
                acc[0] += r0;
                acc[1] += r1;
            } else {
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
                    if (m == pend_mat) acc[m] += r0;
            }
        };
        uint32_t pend_dd[4] = {0u, 0u, 0u, 0u};
        float pend_sx = 0.f;     // Q4_K: the previous unit's sub-block sum of this lane's group of 4
        int pend_sl = 0;         // 8-bit form: the previous unit's table slot
        int k = 0;
        for (int i = set; i < n; i += kSets, ++k) {
            const int u = u0 + i, ug = u / NMAT, mat = u - ug * NMAT, t = ug / G, g = ug - t * G;
            const int s = i % kStages;
            // this lane's eight activations of the group, loaded before the waits
            uint4 xr0 = make_uint4(0u, 0u, 0u, 0u), xr1 = xr0;
            if (loads_x) {
                const int e = g * kGroupK + 8 * xl;
                if (NTOK == 2) {
                    xr0 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + e));
                    xr1 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + p.K + e));
                } else if (p.x_bf16) {
                    xr0 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + e));
                } else {
                    xr0 = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(p.x) + e));
                    xr1 = __ldg(reinterpret_cast<const uint4*>(static_cast<const float*>(p.x) + e + 4));
                }
            }
            const bool got = mbar_wait_bounded(full_bar(bar0, s), (uint32_t)(i / kStages) & 1u, p.fault,
                                               kFaultBulkWaitTimeout);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint32_t src = sbase + (uint32_t)s * kRawStageBytes + raw_row;
            uint32_t v[36];
#pragma unroll
            for (int j = 0; j < 9; ++j) {
                const uint4 w = lds128(src + 16u * (uint32_t)j);
                v[4 * j] = w.x;
                v[4 * j + 1] = w.y;
                v[4 * j + 2] = w.z;
                v[4 * j + 3] = w.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(bar0, s));     // raw rows of stage s read
            uint32_t dd[4];
#pragma unroll
            for (int P = 0; P < 4; ++P) dd[P] = (FMT == kFmtQ4K) ? v[P] : scale_pair(v, P);
            uint32_t c0[32], c1[32];
            // B chunk of a B-writing lane: x_hi and x_lo as bf16, written in the
            // K-half its slot belongs to
            uint4 bhi = make_uint4(0u, 0u, 0u, 0u), blo = bhi;
            float cur_sx = 0.f;
            if (loads_x) {
                if (FMT == kFmtQ4K) {
                    float f[8];
                    if (p.x_bf16) {
                        const uint32_t w4[4] = {xr0.x, xr0.y, xr0.z, xr0.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            f[2 * e] = bf16_lo_to_float(w4[e]);
                            f[2 * e + 1] = bf16_hi_to_float(w4[e]);
                        }
                    } else {
                        f[0] = __uint_as_float(xr0.x); f[1] = __uint_as_float(xr0.y);
                        f[2] = __uint_as_float(xr0.z); f[3] = __uint_as_float(xr0.w);
                        f[4] = __uint_as_float(xr1.x); f[5] = __uint_as_float(xr1.y);
                        f[6] = __uint_as_float(xr1.z); f[7] = __uint_as_float(xr1.w);
                    }
                    cur_sx = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
                }
                if (!bwriter) {
                    // Q4_K lanes outside warp q's B slots: only the sum above
                } else if (NTOK == 2) {
                    bhi = xr0;    // token 0 in the x_hi column, token 1 in the x_lo column
                    blo = xr1;
                } else if (p.x_bf16) {
                    bhi = xr0;
                } else {
                    const float f[8] = {__uint_as_float(xr0.x), __uint_as_float(xr0.y), __uint_as_float(xr0.z),
                                        __uint_as_float(xr0.w), __uint_as_float(xr1.x), __uint_as_float(xr1.y),
                                        __uint_as_float(xr1.z), __uint_as_float(xr1.w)};
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        h[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
                        l[e] = pack_bf16x2(f[2 * e] - bf16_lo_to_float(h[e]), f[2 * e + 1] - bf16_hi_to_float(h[e]));
                    }
                    bhi = make_uint4(h[0], h[1], h[2], h[3]);
                    blo = make_uint4(l[0], l[1], l[2], l[3]);
                }
            }
            if constexpr (FMT == kFmtQ4K) {
                // sub-block sums: lanes 4j .. 4j + 3 hold sub-block j's 32 activations
                cur_sx += __shfl_xor_sync(0xffffffffu, cur_sx, 1);
                cur_sx += __shfl_xor_sync(0xffffffffu, cur_sx, 2);
            }
            // 8-bit form: this unit's group in the table; the B-writing lanes'
            // two pieces of their slot
            int cur_sl = 0;
            uint2 bp0 = make_uint2(0u, 0u), bp1 = bp0;
            if constexpr (F8) {
                cur_sl = g - xg0;
                if (cur_sl < 0) cur_sl += G;
                if (cur_sl >= kXtGroups) cur_sl = 0;       // never: the host checks the table size
                if (bwriter) {
                    const uint4 tq = lds128(sbase + kOffXt + (uint32_t)(cur_sl * 32 + xl) * 16u);
                    bp0 = make_uint2(tq.x, tq.y);
                    bp1 = make_uint2(tq.z, tq.w);
                }
            }
            const uint32_t prev = (uint32_t)(k - 1) & 1u;     // completion parity of the previous unit
            // ---- half 0: K 0..127 (block pairs 0, 1; B atoms 0, 1 written by warps 0, 1)
            if constexpr (F8) codes_pair_e4m3<0>(v, c0);
            else codes_pair<FMT, 0>(v, c0);
            if (k > 0) {
                const bool free = mbar_wait_bounded(aempty_bar(bar0, set, 0), prev, p.fault, kFaultMmaWaitTimeout);
                if (!__all_sync(0xffffffffu, free)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (bwriter && bhalf == 0) {
                if constexpr (F8) {
                    sts64(f8_p0, bp0);
                    sts64(f8_p1, bp1);
                    sts64(f8_n0, make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                    sts64(f8_n1, make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                } else {
                    sts128(b_hi, bhi);
                    sts128(b_lo, blo);
                }
                fence_proxy_async_smem();     // B visible to the tensor core
            }
            tmem_st32(a_taddr, c0);
            if constexpr (F8) codes_pair_e4m3<1>(v, c1);
            else codes_pair<FMT, 1>(v, c1);
            tmem_wait_st();
            tmem_st32(a_taddr + 32u, c1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull_bar(bar0, set, 0));
            // ---- half 1: K 128..255 (block pairs 2, 3; B atoms 2, 3 written by warps 2, 3)
            if constexpr (F8) codes_pair_e4m3<2>(v, c0);
            else codes_pair<FMT, 2>(v, c0);
            if (k > 0) {
                const bool free = mbar_wait_bounded(aempty_bar(bar0, set, 1), prev, p.fault, kFaultMmaWaitTimeout);
                if (!__all_sync(0xffffffffu, free)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (bwriter && bhalf == 1) {
                if constexpr (F8) {
                    sts64(f8_p0, bp0);
                    sts64(f8_p1, bp1);
                    sts64(f8_n0, make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                    sts64(f8_n1, make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                } else {
                    sts128(b_hi, bhi);
                    sts128(b_lo, blo);
                }
                fence_proxy_async_smem();
            }
            tmem_st32(a_taddr + 64u, c0);
            if constexpr (F8) codes_pair_e4m3<3>(v, c1);
            else codes_pair<FMT, 3>(v, c1);
            tmem_wait_st();
            tmem_st32(a_taddr + 96u, c1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull_bar(bar0, set, 1));
            if (k > 0) {
                // the previous unit's D (buffer (k - 1) % 2; complete since its
                // second half's MMAs are), while this unit's MMAs use the other
                uint32_t dv[16];
                tmem_ld16(d_taddr + 16u * prev, dv);
                tmem_wait_ld();
                float r0, r1 = 0.f;
                if constexpr (FMT == kFmtQ4K) r0 = unit_dot_q4k(dv, pend_dd, pend_sx);
                else if constexpr (F8) {
                    float c[8];
                    table_c(sbase, pend_sl, c);
                    r0 = unit_dot_e4m3(dv, pend_dd, c);
                }
                else unit_dot<NTOK>(dv, pend_dd, r0, r1);
                add_unit(r0, r1);
            }
#pragma unroll
            for (int P = 0; P < 4; ++P) pend_dd[P] = dd[P];
            pend_sx = cur_sx;
            pend_sl = cur_sl;
            pend_tile = t;
            pend_mat = mat;
        }
        if (ok && k > 0) {
            // the set's last unit (k - 1)
            const uint32_t last_par = (uint32_t)(k - 1) & 1u;
            const bool fin = mbar_wait_bounded(aempty_bar(bar0, set, 1), last_par, p.fault, kFaultMmaWaitTimeout);
            if (__all_sync(0xffffffffu, fin)) {
                tc_fence_after();
                uint32_t dv[16];
                tmem_ld16(d_taddr + 16u * last_par, dv);
                tmem_wait_ld();
                float r0, r1 = 0.f;
                if constexpr (FMT == kFmtQ4K) r0 = unit_dot_q4k(dv, pend_dd, pend_sx);
                else if constexpr (F8) {
                    float c[8];
                    table_c(sbase, pend_sl, c);
                    r0 = unit_dot_e4m3(dv, pend_dd, c);
                }
                else unit_dot<NTOK>(dv, pend_dd, r0, r1);
                add_unit(r0, r1);
            }
        }
        if (acc_tile >= 0)
#pragma unroll
            for (int m = 0; m < NCH; ++m) part[part_at(set, acc_tile - tile0, m, row)] = acc[m];
        if (!counted) count_in();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // no MMA may still be writing TMEM when it is released
        const uint32_t tmem = *tmem_slot;
        mbar_wait_bounded(done_bar(bar0), 0u, p.fault, kFaultMmaWaitTimeout);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
    }
    if (n <= 0) return;

    // ---------------- the range's tiles: whole ones -> y; the last one, when
    // this CTA covers its first unit but not its last, is finished here
    const int tile1 = (u1 - 1) / GU;
    const bool fin1 = (tile1 + 1) * GU > u1 && tile1 * GU >= u0;
    const int r = threadIdx.x;
    if (r < kTileRows) {
        for (int t = tile0; t <= tile1; ++t) {
            if (t == tile0 && contrib0) continue;                 // published already
            const int lt = t - tile0;
            float v[NCH];
#pragma unroll
            for (int m = 0; m < NCH; ++m)
                v[m] = part[part_at(0, lt, m, r)] + part[part_at(1, lt, m, r)] + part[part_at(2, lt, m, r)];
            if (t == tile1 && fin1) {
                const int c_last = owner_of((t + 1) * GU - 1, p.units, ctas);
                for (int c = cta + 1; c <= c_last; ++c)
#pragma unroll
                    for (int m = 0; m < NCH; ++m) {
                        unsigned long long* src = share + ((size_t)c * 2 + m) * kTileRows + r;
                        const unsigned long long w = wait_tagged_u64(src, p.fault, kFaultShareWaitTimeout);
                        v[m] += __uint_as_float((uint32_t)w);
                        st_relaxed_u64(src, 0ull);                 // consumed
                    }
            }
            const int64_t yrow = (int64_t)t * kTileRows + r;
            if (yrow < p.N) {
                if constexpr (NTOK == 2) {
                    if (p.y_bf16) {
                        store_out<__nv_bfloat16>(p.y, yrow, v[0]);
                        store_out<__nv_bfloat16>(p.y, (int64_t)p.N + yrow, v[1]);
                    } else {
                        store_out<float>(p.y, yrow, v[0]);
                        store_out<float>(p.y, (int64_t)p.N + yrow, v[1]);
                    }
                } else {
                    float o = v[0];
                    if constexpr (NMAT == 2) o = gelu_tanh(v[0]) * v[1];
                    if (p.y_bf16) store_out<__nv_bfloat16>(p.y, yrow, o);
                    else store_out<float>(p.y, yrow, o);
                }
            }
        }
    }
}

template <int NMAT, int NTOK>
__global__ void __launch_bounds__(kThreads, 1) qmv_q4_0_tc_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4, NMAT, NTOK, false>(p);
}

// bf16 activations, one token: the 8-bit operand form
template <int NMAT>
__global__ void __launch_bounds__(kThreads, 1) qmv_q4_0_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4, NMAT, 1, true>(p);
}

__global__ void __launch_bounds__(kThreads, 1) qmv_q4_k_tc_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4K, 1, 1, false>(p);
}

}  // namespace

// The tensor-core M = 1 path takes K % 256 == 0, at most kQtcMaxTiles tiles
// and kQtcMaxCtas CTAs, and unit ranges that span at most kMaxLocalTiles
// tiles per CTA.
bool qmv_tc_supported(int nmat, int64_t N, int64_t K, int sm_count) {
    if (nmat < 1 || nmat > 2) return false;
    if (K % kGroupK != 0 || K < kGroupK || N < 1 || sm_count < 1 || sm_count > kQtcMaxCtas) return false;
    const int64_t tiles = (N + kTileRows - 1) / kTileRows;
    if (tiles > kQtcMaxTiles) return false;
    const int64_t per_tile = (K / kGroupK) * nmat;
    const int64_t units = tiles * per_tile;
    if (units > INT32_MAX) return false;
    const int64_t ctas = units < sm_count ? units : sm_count;
    const int64_t per = (units + ctas - 1) / ctas;
    return per / per_tile + 2 <= kMaxLocalTiles;
}

size_t qmv_tc_smem_bytes() { return kSmemBytes; }

// fmt: kFmtQ4 or kFmtQ4K (one matrix, one token).  nmat = 2: gate + up (one
// token).  ntok = 2 (nmat = 1, bf16 X of two rows of K, Y of two rows of N):
// two tokens.
cudaError_t launch_qmv_tc(int fmt, int nmat, int ntok, const CUtensorMap* tmap_w, const void* x, int x_bf16,
                          void* y, int y_bf16, int N, int K, int sm_count, unsigned int* fault, cudaStream_t stream) {
    static std::atomic<unsigned int> calls{0};
    if (nmat * ntok > 2 || (ntok == 2 && !x_bf16)) return cudaErrorInvalidValue;
    if (fmt == kFmtQ4K && nmat * ntok != 1) return cudaErrorInvalidValue;
    QtcParams p;
    p.tmap_w[0] = tmap_w[0];
    p.tmap_w[1] = tmap_w[nmat == 2 ? 1 : 0];
    p.x = x;
    p.y = y;
    p.fault = fault;
    p.N = N;
    p.K = K;
    p.tiles = (N + kTileRows - 1) / kTileRows;
    p.groups = K / kGroupK;
    p.units = p.tiles * p.groups * nmat;
    p.slot = (int)(calls.fetch_add(1u) % kQtcSlots);
    p.x_bf16 = x_bf16;
    p.y_bf16 = y_bf16;
    const int ctas = p.units < sm_count ? p.units : sm_count;
    // the 8-bit form needs every K-group of a CTA's unit range in its table
    const int per_cta = (p.units + ctas - 1) / ctas;
    const bool f8 = fmt == kFmtQ4 && ntok == 1 && x_bf16 &&
                    std::min(p.groups, (per_cta - 1) / nmat + 2) <= kXtGroups;
    auto kernel = fmt == kFmtQ4K ? qmv_q4_k_tc_kernel
                  : f8           ? (nmat == 2 ? qmv_q4_0_tc_e4m3_kernel<2> : qmv_q4_0_tc_e4m3_kernel<1>)
                  : (nmat == 2 ? qmv_q4_0_tc_kernel<2, 1>
                               : (ntok == 2 ? qmv_q4_0_tc_kernel<1, 2> : qmv_q4_0_tc_kernel<1, 1>));
    static thread_local int prepared_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (prepared_device != dev) {
        for (auto f : {qmv_q4_0_tc_kernel<1, 1>, qmv_q4_0_tc_kernel<2, 1>, qmv_q4_0_tc_kernel<1, 2>,
                       qmv_q4_0_tc_e4m3_kernel<1>, qmv_q4_0_tc_e4m3_kernel<2>, qmv_q4_k_tc_kernel}) {
            cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
            if (e != cudaSuccess) return e;
        }
        prepared_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace qbw
