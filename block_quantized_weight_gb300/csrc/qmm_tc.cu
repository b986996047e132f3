// qmm_tc.cu -- the small-M Q4_0 product Y[M, N] = X[M, K] W[N, K]^T on the
// fifth-generation tensor cores (tcgen05), M <= 32 token rows.
//
// One CTA computes a tile of 128 weight rows over a range of K (split K):
//   * D = W_tile X^T is a 128 x NT fp32 accumulator in tensor memory (TMEM),
//     NT = M rounded up to 16 (the MMA's N);
//   * the A operand (128 weight rows x 16 K per MMA, bf16) is written to TMEM
//     by the dequantizing warps themselves (tcgen05.st): a thread owns one
//     weight row = one TMEM lane, so dequantized weights never touch shared
//     memory;
//   * the B operand (NT token rows x K, bf16) arrives in shared memory by TMA
//     with the 128-byte swizzle the MMA's K-major descriptor expects; token
//     rows past M read as zeros;
//   * raw Q4_0 bytes arrive by TMA in K-groups of 256 (8 blocks = 144 bytes
//     per row), a box of 128 rows x 144 bytes.
//
// Warp roles: three sets of four dequantizing warps (warps 0..11).  Set g
// takes the CTA's K-groups g, g + 3, g + 6, ... and owns TMEM A stage g;
// warp 4g + q of the set handles rows 32q .. 32q + 31 (the TMEM lanes of its
// quarter) over the whole group.  Warp 12 lane 0 issues the TMA copies.
// Warps 13, 14 and 15 (lane 0) issue the MMAs: issuer j takes set j's groups
// (all 16 K-steps of each) into its own accumulator D_j.  A group's A stage is
// published in two halves of 128 K, each with its own pair of mbarriers, so
// the MMAs on the first half run while the set decodes the second.  One thread issues a
// narrow (N <= 32) MMA only about every 50 cycles, well below what the tensor
// core retires, and issuing threads overlap, so three issuers keep up with
// three sets.  Warps 0..3 read D_0 + D_1 + D_2 back.
//
// Dequantization to bf16, two adjacent weights j, j + 1 of a block at a time:
// a byte permute puts qs[j] and qs[j + 1] in bytes 0 and 2 of a word; a LOP3
// keeps their low nibbles and ORs in the bf16 exponent of 128, which gives
// the pair (128 + c_j, 128 + c_j+1) exactly; the same after a 4-bit shift
// gives codes j + 16 and j + 17.  A packed bf16 add of -136 leaves the exact
// integers c - 8.  The block's fp16 scale d is carried as two bf16 parts, d_hi = bf16(d) and
// d_lo = bf16(d - d_hi), and the weight is fma(c - 8, d_hi, (c - 8) d_lo),
// rounded once to bf16.  The argument of that final rounding is within about
// 2^-15 of (c - 8) d relative (d_lo's own rounding and that of the small
// product), so each weight is within 2^-8 (1 + 2^-7) of its exact value
// relative: one rounding to 8 significant bits, well inside the 1e-2 bound
// on sum |w x| of the tensor-core path.
//
// Split K, two ways.  With at most 8 splits per tile, the splits of a tile run
// as one thread-block cluster: each CTA leaves its partial tile (128 rows x M,
// M padded to 4) in its own shared memory, which the pipeline no longer needs
// once the last MMA has completed; after a cluster barrier each CTA sums a
// slice of the tile over all CTAs of the cluster (distributed shared memory),
// in split order, and writes it to Y; a second cluster barrier keeps every
// CTA's shared memory alive until its peers have read it.  With more splits,
// each CTA writes its partial tile to the workspace; the last CTA of a tile
// (counted with an atomic) adds the partials in split order and writes Y,
// then resets the counter and clears the partials, so the workspace is all
// zero again after every call.
//
// Stream-K (M <= 16).  Where whole-tile splits leave SMs idle (42 tiles of 3
// splits use 126 of 152) and K is long (16 groups or more a CTA), one CTA per
// SM takes an equal range of the (tile, K-group) units in tile-major order
// instead.  A range meets at most two tiles (it is never longer than a tile),
// so a CTA has one or two segments, each with its own three accumulators
// (TMEM 384 + 2 x 3 x 16 columns).  A segment that starts inside a tile is a
// share: the CTA publishes it at the end of its range as one tagged 64-bit
// word (fp32 bits, tag) per row and token column, the tag being the launch's
// own (launch_tag: derived from the grid id), so a word left by another call
// is never taken.  The CTA that covers a tile's first group finishes the tile
// at the end of its range: it adds the later CTAs' shares after its own, in
// CTA order, clears them and writes Y.  A range covering a whole tile writes Y directly.  Results depend
// only on the plan, so they are bit-reproducible.
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"
#include "tc_common.cuh"

namespace qbw {
namespace {

using namespace tc;

constexpr int kTileRows = 128;
constexpr int kGroupK = 256;                  // K per pipeline stage (8 Q4_0 blocks)
constexpr int kGroupBytes = 144;              // raw bytes per row per K-group
constexpr int kSets = 3;                      // dequantizing warp sets = TMEM A stages
constexpr int kDequantWarps = 4 * kSets;
constexpr int kProducerWarp = kDequantWarps;
constexpr int kMmaWarp0 = kDequantWarps + 1;  // issuer j: warp kMmaWarp0 + j
constexpr int kIssuers = kSets;               // one per set
constexpr int kThreads = (kDequantWarps + 1 + kIssuers) * 32;
constexpr int kStages = 6;                    // shared-memory stages (raw W + X)
constexpr int kAStages = kSets;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColsPerStage = kGroupK / 2;          // 2 bf16 per 32-bit column
constexpr uint32_t kDCol = kAStages * kAColsPerStage;     // accumulator D_j of segment s at kDCol + NT (3 s + j)
constexpr uint32_t kRawStageBytes = kTileRows * kGroupBytes;   // 18432
constexpr int kReduceItems = 3;               // row x 4-column items per thread in the split-K sum: 480 x 3 >= 128 x 8

// bf16x2 constant: (-136, -136)
constexpr uint32_t kBf16Minus136 = 0xC308C308u;

// (128 + c) pair -> d (c - 8) pair: (t - 136) is the exact integer c - 8, the
// product with d_lo is rounded (tiny), and the fma with d_hi rounds the weight
// once.
__device__ __forceinline__ uint32_t scale_pair(uint32_t t, uint32_t dhi, uint32_t dlo, uint32_t m136) {
    uint32_t c, lo, r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(t), "r"(m136));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(c), "r"(dlo));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(c), "r"(dhi), "r"(lo));
    return r;
}

// One Q4_0 block of a row whose 144 bytes of the K-group are the words v[].
// OFF is the byte offset of the block's qs[0]; the fp16 scale is half SH of
// word SW.  Writes the block's 16 bf16x2 columns in K order: column t holds
// elements 2t (low half) and 2t + 1 (high half).
template <int OFF, int SW, int SH>
__device__ __forceinline__ void dequant_block(const uint32_t (&v)[36], uint32_t* col) {
    const uint32_t dbits = SH ? (v[SW] >> 16) : (v[SW] & 0xFFFFu);
    const float d = half_bits_to_float(dbits);
    const uint32_t m136 = kBf16Minus136;
    uint32_t dhi, dlo;
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(dhi) : "f"(d));
    const float rest = d - __uint_as_float(dhi << 16);     // exact in fp32
    asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(dlo) : "f"(rest));
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        // qs[j] and qs[j + 1] share a word: OFF + j is even and OFF % 4 is 0 or 2
        const int byte = OFF + j;
        uint32_t lo, hi;
        if ((byte & 3) == 0) nibble_pairs<0>(v[byte >> 2], lo, hi);
        else nibble_pairs<2>(v[byte >> 2], lo, hi);
        col[j >> 1] = scale_pair(lo, dhi, dlo, m136);         // elements j, j + 1
        col[8 + (j >> 1)] = scale_pair(hi, dhi, dlo, m136);   // elements 16 + j, 17 + j
    }
}

// Block pair P (blocks 2P, 2P + 1) of the row's K-group -> 32 columns.  Pair
// P starts at byte 36P: scale A in the low half of word 9P, qs A from byte
// 36P + 2, scale B in the high half of word 9P + 4, qs B from byte 36P + 20.
template <int P>
__device__ __forceinline__ void dequant_pair(const uint32_t (&v)[36], uint32_t (&col)[32]) {
    dequant_block<36 * P + 2, 9 * P, 0>(v, col);
    dequant_block<36 * P + 20, 9 * P + 4, 1>(v, col + 16);
}

struct QmmParams {
    CUtensorMap tmap_w;     // Q4_0 rows as 8-byte words, box (18, 128)
    CUtensorMap tmap_x;     // X [M][K] bf16, box (64, NT), 128-byte swizzle
    void* y;
    float* partials;        // [splits][tiles][128][M rounded up to 4] fp32 (splits > 1)
    unsigned int* counters; // [tiles] (splits > 1)
    unsigned long long* share;   // stream-K: [ctas][M rounded up to 4][128] tagged words
    unsigned int* fault;
    int32_t M, N, K;
    int32_t NT;             // MMA N: M rounded up to 16
    int32_t groups;         // K / 256
    int32_t splits;
    int32_t tiles;          // ceil(N / 128)
    int32_t y_bf16;
    int32_t cluster;        // 1: the splits of a tile are one cluster (no workspace)
    int32_t streamk;        // 1: ctas CTAs over `units` (tile, group) units (NT = 16)
    int32_t ctas;
    int32_t units;          // tiles * groups
};

// Barrier layout shared by every role: full[kStages], empty[kStages],
// afull[kAStages][2], aempty[kAStages][2] (per half of the group's K), dfull,
// 8 bytes each from bar0.
constexpr int kBarriers = 2 * kStages + 4 * kAStages + 1;
__device__ __forceinline__ uint32_t full_bar_at(uint32_t bar0, int s) { return bar0 + 8u * (uint32_t)s; }
__device__ __forceinline__ uint32_t empty_bar_at(uint32_t bar0, int s) { return bar0 + 8u * (uint32_t)(kStages + s); }
__device__ __forceinline__ uint32_t afull_bar_at(uint32_t bar0, int a, int h) {
    return bar0 + 8u * (uint32_t)(2 * kStages + 2 * a + h);
}
__device__ __forceinline__ uint32_t aempty_bar_at(uint32_t bar0, int a, int h) {
    return bar0 + 8u * (uint32_t)(2 * kStages + 2 * kAStages + 2 * a + h);
}
__device__ __forceinline__ uint32_t dfull_bar_at(uint32_t bar0) {
    return bar0 + 8u * (uint32_t)(2 * kStages + 4 * kAStages);
}

// v[q] = sum of the included accumulators' column q (16 columns from taddr;
// D_1 and D_2 at nt and 2 nt columns further), added in issuer order.
__device__ __forceinline__ void read_d(uint32_t taddr, uint32_t nt, bool i0, bool i1, bool i2, float (&v)[16]) {
    uint32_t d0[16], d1[16], d2[16];
    tmem_ld16(taddr, d0);
    tmem_ld16(taddr + nt, d1);
    tmem_ld16(taddr + 2u * nt, d2);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 16; ++q)
        v[q] = ((i0 ? __uint_as_float(d0[q]) : 0.f) + (i1 ? __uint_as_float(d1[q]) : 0.f)) +
               (i2 ? __uint_as_float(d2[q]) : 0.f);
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

// A row's share: token column q at dst[128 q], as (fp32 bits, this launch's
// tag), so that a finisher never takes a word left by another call.
__device__ __forceinline__ void store_share(unsigned long long* dst, const float (&v)[16], int mp) {
    const unsigned long long tag = (unsigned long long)launch_tag() << 32;
#pragma unroll
    for (int q = 0; q < 16; ++q)
        if (q < mp) st_relaxed_u64(dst + (size_t)q * kTileRows, tag | (unsigned long long)__float_as_uint(v[q]));
}

// One dequantizing warp of set g over the CTA's K-groups g, g + 3, ...
// Per group: wait for the raw stage; read the lane's 144 bytes with nine
// 16-byte loads (8 consecutive lanes = 8 rows 144 bytes apart hit 8 distinct
// 16-byte bank groups: conflict-free); release the stage; decode the four
// block pairs into two alternating register buffers and store each into TMEM
// A stage g.  A buffer is rewritten only after a tcgen05.wait::st covering
// its previous store.  raw_row: the row's byte offset within a stage;
// a_taddr: TMEM address of the quarter's lanes, A stage g, column 0.
__device__ __forceinline__ bool dequant_warp(int g, uint32_t raw_row, uint32_t a_taddr, uint32_t sbase,
                                             uint32_t stage_bytes, uint32_t bar0, int lane, int ng,
                                             unsigned int* fault) {
    for (int i = g; i < ng; i += kSets) {
        const int s = i % kStages;
        const bool got = mbar_wait_bounded(full_bar_at(bar0, s), (uint32_t)(i / kStages) & 1u, fault,
                                           kFaultBulkWaitTimeout);
        if (!__all_sync(0xffffffffu, got)) return false;
        const uint32_t src = sbase + (uint32_t)s * stage_bytes + raw_row;
        uint32_t v[36];
#pragma unroll
        for (int j = 0; j < 9; ++j) {
            const uint4 q = lds128(src + 16u * (uint32_t)j);
            v[4 * j] = q.x;
            v[4 * j + 1] = q.y;
            v[4 * j + 2] = q.z;
            v[4 * j + 3] = q.w;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar_at(bar0, s));     // raw W of stage s read
        uint32_t c0[32], c1[32];
        const uint32_t par = (uint32_t)((i / kSets) - 1) & 1u;
        // ---- first half of the group's K (block pairs 0, 1): the MMAs on it
        // run while the second half is decoded
        dequant_pair<0>(v, c0);
        if (i >= kSets) {
            // the MMAs of group i - 3 have finished reading this half of A stage g
            const bool free = mbar_wait_bounded(aempty_bar_at(bar0, g, 0), par, fault, kFaultMmaWaitTimeout);
            if (!__all_sync(0xffffffffu, free)) return false;
            tc_fence_after();
        }
        tmem_st32(a_taddr, c0);
        dequant_pair<1>(v, c1);
        tmem_wait_st();
        tmem_st32(a_taddr + 32u, c1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull_bar_at(bar0, g, 0));
        // ---- second half (block pairs 2, 3)
        dequant_pair<2>(v, c0);
        if (i >= kSets) {
            const bool free = mbar_wait_bounded(aempty_bar_at(bar0, g, 1), par, fault, kFaultMmaWaitTimeout);
            if (!__all_sync(0xffffffffu, free)) return false;
            tc_fence_after();
        }
        tmem_st32(a_taddr + 64u, c0);
        dequant_pair<3>(v, c1);
        tmem_wait_st();
        tmem_st32(a_taddr + 96u, c1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull_bar_at(bar0, g, 1));
    }
    return true;
}

// One MMA issuer (lane 0 of its warp): all 16 K-steps of set J's groups J,
// J + 3, ... of the CTA's ng K-groups, into accumulator D_J of the group's
// segment (groups below nA: the first; the rest: the second).  Every operand
// of a group's MMAs is formed before its barrier waits, and stage and phase
// are carried incrementally, so that once the A stage is published the MMAs
// go out back to back: this thread shares its SM sub-partition with three
// busy dequantizing warps, and every instruction between two MMAs costs
// issue slots.
template <int J, bool SK>
__device__ __forceinline__ bool issue_mmas(uint32_t tmem, uint32_t sbase, uint32_t stage_bytes, uint32_t bar0, int nt,
                                           int ng, int nA, unsigned int* fault) {
    constexpr int kSteps = kGroupK / 16;                     // 16 MMAs per group
    const uint32_t idesc = idesc_bf16(kTileRows, nt);
    const uint32_t d_seg0 = tmem + kDCol + (uint32_t)nt * (uint32_t)J;
    const uint32_t d_seg1 = d_seg0 + 3u * (uint32_t)nt;
    const uint32_t a_tmem = tmem + (uint32_t)J * kAColsPerStage;   // set J's A stage
    // X of stage s, atom t, 16-element slice c: descriptor start field advances
    // by stage_bytes / 16, nt * 128 / 16 and 32 / 16 respectively
    const uint64_t atom_step = (uint64_t)((uint32_t)nt * 8u);
    const uint64_t stage_step = (uint64_t)(stage_bytes >> 4);
    uint64_t koff[kSteps];
#pragma unroll
    for (int k = 0; k < kSteps; ++k) koff[k] = (uint64_t)(k >> 2) * atom_step + (uint64_t)((k & 3) * 2);
    // group i = J + 3 t sits in stage i % 6, pass i / 6, and uses A stage J for
    // the t-th time
    const uint64_t ds0 = sw128_desc(sbase + kRawStageBytes);
    uint32_t aphase = 0;
    bool ok = true;
    for (int i = J; i < ng; i += kSets) {
        const int s = i % kStages;
        const uint32_t sphase = (uint32_t)(i / kStages) & 1u;
        const uint64_t ds = ds0 + (uint64_t)s * stage_step;
        const bool seg1 = SK && i >= nA;
        const uint32_t d_tmem = seg1 ? d_seg1 : d_seg0;
        const uint32_t acc0 = (seg1 ? i - kSets >= nA : i > J) ? 1u : 0u;
        ok = mbar_wait_bounded(full_bar_at(bar0, s), sphase, fault, kFaultMmaWaitTimeout) &&
             mbar_wait_bounded(afull_bar_at(bar0, J, 0), aphase, fault, kFaultMmaWaitTimeout);
        if (!ok) break;
        tc_fence_after();
        tc_mma(d_tmem, a_tmem, ds + koff[0], idesc, acc0);
#pragma unroll
        for (int k = 1; k < kSteps / 2; ++k) tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, ds + koff[k], idesc, 1u);
        tc_commit(aempty_bar_at(bar0, J, 0));     // first half of TMEM A stage J consumed
        ok = mbar_wait_bounded(afull_bar_at(bar0, J, 1), aphase, fault, kFaultMmaWaitTimeout);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = kSteps / 2; k < kSteps; ++k) tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, ds + koff[k], idesc, 1u);
        tc_commit(empty_bar_at(bar0, s));         // X tile of stage s consumed
        tc_commit(aempty_bar_at(bar0, J, 1));     // second half consumed
        aphase ^= 1u;
    }
    // completes when every MMA issued above has finished, even after a
    // timeout (the accumulator is then not read, only TMEM released)
    tc_commit(dfull_bar_at(bar0));
    return ok;
}


__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_f4(uint32_t a, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// 16 bytes at shared-memory address `a` of the cluster's CTA `rank`
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t a, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra) : "memory");
    return v;
}

// SK: a stream-K plan (p.streamk = 1); the split-K plans compile without its code.
template <bool SK>
__global__ void __launch_bounds__(kThreads, 1) qmm_q4_0_tc_kernel(const __grid_constant__ QmmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The CTA's ng K-groups: groups g_begin .. g_begin + nA - 1 of `tile`, then
    // (stream-K only) groups 0 .. ng - nA - 1 of tile + 1.
    int tile, split, g_begin, ng, nA;
    if constexpr (SK) {
        const int u0 = (int)((int64_t)p.units * blockIdx.x / p.ctas);
        const int u1 = (int)((int64_t)p.units * (blockIdx.x + 1) / p.ctas);
        tile = u0 / p.groups;
        g_begin = u0 - tile * p.groups;
        split = 0;
        ng = u1 - u0;
        nA = min(ng, p.groups - g_begin);
        // the plan keeps NT = 16 (the two segments' accumulators fit TMEM) and
        // every range non-empty and no longer than a tile
        if (p.NT != 16 || ng < 1 || ng > p.groups) {
            if (threadIdx.x == 0) record_fault(p.fault, kFaultPlan);
            return;
        }
    } else {
        tile = blockIdx.x / p.splits;
        split = blockIdx.x - tile * p.splits;
        g_begin = (int)((int64_t)p.groups * split / p.splits);
        ng = (int)((int64_t)p.groups * (split + 1) / p.splits) - g_begin;
        nA = ng;
    }
    const bool two = SK && nA < ng;
    // the last segment: its tile, first group there and length; a stream-K
    // CTA that covers a tile's first group but not all of it finishes the tile
    const int tile_e = two ? tile + 1 : tile;
    const int start_e = two ? 0 : g_begin;
    const int len_e = ng - (two ? nA : 0);
    const bool finisher = SK && start_e == 0 && len_e < p.groups;

    // shared memory: [stages][raw W 18432 B | X NT x 256 bf16] (1024-aligned), barriers, TMEM slot
    const uint32_t xbytes = (uint32_t)p.NT * kGroupK * 2;            // 4 swizzle atoms of NT x 128 B
    const uint32_t stage_bytes = kRawStageBytes + xbytes;            // multiple of 1024
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kStages * stage_bytes;
    const uint32_t dfull_bar = dfull_bar_at(bar0);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kStages * stage_bytes + 8 * kBarriers);
    bool ok = true;

    // K-group i of this CTA -> stage i % kStages: raw W box and the 4 X boxes
    auto issue_w = [&](int i) {
        const int s = i % kStages;
        mbar_arrive_expect_tx(full_bar_at(bar0, s), kRawStageBytes + xbytes);
        const bool seg1 = SK && i >= nA;
        tma_load_2d(sbase + (uint32_t)s * stage_bytes, &p.tmap_w, (seg1 ? i - nA : g_begin + i) * (kGroupBytes / 8),
                    (seg1 ? tile + 1 : tile) * kTileRows, full_bar_at(bar0, s), policy_evict_first());
    };
    auto issue_x = [&](int i) {
        const uint32_t st = sbase + (uint32_t)(i % kStages) * stage_bytes;
#pragma unroll
        for (int a = 0; a < 4; ++a)
            tma_load_2d(st + kRawStageBytes + (uint32_t)a * (uint32_t)p.NT * 128u, &p.tmap_x,
                        ((SK && i >= nA) ? i - nA : g_begin + i) * kGroupK + a * 64, 0, full_bar_at(bar0, i % kStages),
                        0ull);
    };

    // The producer initialises the barriers, releases everyone else through
    // named barrier 1 without waiting there itself, and starts the first
    // copies while warp 0 allocates TMEM.
    if (warp == kProducerWarp) {
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(full_bar_at(bar0, s), 1);
                mbar_init(empty_bar_at(bar0, s), 4 + 1);   // the group's 4 dequantizing warps + its issuer's commit
            }
            for (int a = 0; a < kAStages; ++a)
                for (int h = 0; h < 2; ++h) {
                    mbar_init(afull_bar_at(bar0, a, h), 4);
                    mbar_init(aempty_bar_at(bar0, a, h), 1);
                }
            mbar_init(dfull_bar, kIssuers);
            fence_mbar_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 1, %0;" ::"n"(kThreads) : "memory");
        if (lane == 0) {
            prefetch_tmap(&p.tmap_w);
            prefetch_tmap(&p.tmap_x);
            // the weights do not depend on the preceding grid: the first stages'
            // weight boxes go out before its completion, X after
            const int pre = ng < kStages ? ng : kStages;
            for (int i = 0; i < pre; ++i) issue_w(i);
            grid_dependency_wait();
            for (int i = 0; i < pre; ++i) issue_x(i);
            for (int i = pre; i < ng && ok; ++i) {
                const int s = i % kStages;
                ok = mbar_wait_bounded(empty_bar_at(bar0, s), (uint32_t)((i / kStages) - 1) & 1u, p.fault,
                                       kFaultBulkWaitTimeout);
                if (ok) {
                    issue_w(i);
                    issue_x(i);
                }
            }
        }
    } else {
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "n"(kTmemCols));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
        tc_fence_after();
    }
    // X, Y and the workspace belong to the preceding grid's stream order
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp >= kMmaWarp0) {
        // ---------------- MMA issuers: issuer j takes set j's groups
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            if (warp == kMmaWarp0) ok = issue_mmas<0, SK>(tmem, sbase, stage_bytes, bar0, p.NT, ng, nA, p.fault);
            else if (warp == kMmaWarp0 + 1) ok = issue_mmas<1, SK>(tmem, sbase, stage_bytes, bar0, p.NT, ng, nA, p.fault);
            else ok = issue_mmas<2, SK>(tmem, sbase, stage_bytes, bar0, p.NT, ng, nA, p.fault);
        }
    } else if (warp < kDequantWarps) {
        // ---------------- dequantizing warps
        const uint32_t tmem = *tmem_slot;
        const int set = warp >> 2, quarter = warp & 3;   // TMEM lanes 32 quarter .. +31
        const int row = quarter * 32 + lane;             // weight row within the tile
        ok = dequant_warp(set, (uint32_t)row * kGroupBytes,
                          tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)set * kAColsPerStage, sbase,
                          stage_bytes, bar0, lane, ng, p.fault);
        // ---------------- epilogue: warps 0..3 read the last segment's D_0 + D_1 + D_2
        // (128 rows x NT) and emit
        if (warp < 4) {
            const bool got = ok && mbar_wait_bounded(dfull_bar, 0u, p.fault, kFaultMmaWaitTimeout);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                const int n = tile_e * kTileRows + row;
                // issuer j has groups in the last segment (D_j holds nothing otherwise)
                bool inc[kSets];
#pragma unroll
                for (int j = 0; j < kSets; ++j) inc[j] = two ? (j - nA % kSets + kSets) % kSets < len_e : j < ng;
                const int mp = (p.M + 3) & ~3;
                float* part = p.partials + ((size_t)(split * p.tiles + tile) * kTileRows + row) * (size_t)mp;
                if constexpr (SK)
                    if (two) {
                        // the first segment is a share of a tile that an earlier CTA
                        // finishes; published here, at the end of the range (a
                        // mid-range publish held up the decode and measured slower)
                        float v0[16];
                        read_d(tmem + ((uint32_t)(quarter * 32) << 16) + kDCol, 16u, true, nA > 1, nA > 2, v0);
                        store_share(p.share + (size_t)blockIdx.x * mp * kTileRows + row, v0, mp);
                    }
                const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + kDCol + (two ? 3u * p.NT : 0u);
                for (int c0 = 0; c0 < p.NT; c0 += 16) {
                    float v[16];
                    read_d(lane_base + (uint32_t)c0, (uint32_t)p.NT, inc[0], inc[1], inc[2], v);
                    bool to_y = p.splits == 1;
                    if constexpr (SK) {
                        if (start_e > 0) {
                            // a share of a tile that an earlier CTA finishes
                            store_share(p.share + (size_t)blockIdx.x * mp * kTileRows + row, v, mp);
                            to_y = false;
                        } else if (finisher) {
                            // the CTA's own part, [column][row] in shared memory (the
                            // pipeline's stages are idle once every MMA has completed);
                            // all warps finish the tile below
                            float* own = reinterpret_cast<float*>(smem);
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                if (q < mp) own[q * kTileRows + row] = v[q];
                            to_y = false;
                        }
                    }
                    if (to_y) {
                        if (n < p.N) {
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const int m = c0 + q;
                                if (m < p.M) {
                                    if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, v[q]);
                                    else store_out<float>(p.y, (int64_t)m * p.N + n, v[q]);
                                }
                            }
                        }
                    } else if (SK) {
                        // published or left for the finish above
                    } else if (p.cluster) {
                        // column quad u of this row at byte (u * 128 + row) * 16 of
                        // the CTA's shared memory: a warp stores 512 contiguous bytes
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (c0 + q < mp)
                                st_shared_f4(sbase + (uint32_t)(((c0 + q) / 4 * kTileRows + row) * 16),
                                             make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]));
                    } else {
                        // this row's columns c0 .. c0 + 15 below mp, as 16-byte vectors
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (c0 + q < mp)
                                *reinterpret_cast<float4*>(part + c0 + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
                    }
                }
                if (p.splits > 1 && !p.cluster) __threadfence();   // partials visible before the split counter moves
            } else {
                ok = false;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // no MMA may still be writing TMEM when it is released
        const uint32_t tmem = *tmem_slot;
        mbar_wait_bounded(dfull_bar, 0u, p.fault, kFaultMmaWaitTimeout);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
    }

    if constexpr (SK) {
        if (finisher) {
            // Finish the tile: word t = column t / 128, row t % 128 of the CTA's own
            // part plus, in CTA order, the shares of the later CTAs whose ranges
            // start inside the tile.  Up to four shares' words are loaded at once;
            // a word not yet tagged is waited for (after one timeout, no longer),
            // and every word read is cleared.
            const int mp = (p.M + 3) & ~3;
            const int words = kTileRows * mp;
            const uint32_t tag = launch_tag();
            const int tile_end_unit = (tile_e + 1) * p.groups;
            int c_end = (int)blockIdx.x + 1;
            while (c_end < p.ctas && (int)((int64_t)p.units * c_end / p.ctas) < tile_end_unit) ++c_end;
            const float* own = reinterpret_cast<const float*>(smem);
            constexpr int kWordsPerThread = 16 * kTileRows / kThreads;   // mp <= 16
            float acc[kWordsPerThread];
#pragma unroll
            for (int k = 0; k < kWordsPerThread; ++k) {
                const int t = (int)threadIdx.x + k * kThreads;
                acc[k] = t < words ? own[t] : 0.f;
            }
            bool live = true;
            for (int c0 = (int)blockIdx.x + 1; c0 < c_end; c0 += 4) {
                unsigned long long w[4][kWordsPerThread];
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int k = 0; k < kWordsPerThread; ++k) {
                        const int t = (int)threadIdx.x + k * kThreads;
                        w[u][k] = (c0 + u < c_end && t < words)
                                      ? ld_relaxed_u64(p.share + (size_t)(c0 + u) * words + t)
                                      : 0ull;
                    }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int k = 0; k < kWordsPerThread; ++k) {
                        const int t = (int)threadIdx.x + k * kThreads;
                        if (c0 + u < c_end && t < words) {
                            unsigned long long* src = p.share + (size_t)(c0 + u) * words + t;
                            unsigned long long wk = w[u][k];
                            if ((uint32_t)(wk >> 32) != tag) {
                                wk = wait_tag_u64(src, tag, p.fault, kFaultShareWaitTimeout, live ? kWaitLimitNs : 0);
                                live = live && (uint32_t)(wk >> 32) == tag;
                            }
                            acc[k] += __uint_as_float((uint32_t)wk);
                            st_relaxed_u64(src, 0ull);
                        }
                    }
            }
#pragma unroll
            for (int k = 0; k < kWordsPerThread; ++k) {
                const int t = (int)threadIdx.x + k * kThreads;
                const int m = t / kTileRows, n = tile_e * kTileRows + (t & (kTileRows - 1));
                if (t < words && m < p.M && n < p.N) {
                    if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, acc[k]);
                    else store_out<float>(p.y, (int64_t)m * p.N + n, acc[k]);
                }
            }
        }
        return;
    }

    if (p.splits > 1 && p.cluster) {
        // every partial tile of the cluster is in place after this barrier
        cluster_sync_all();
        const int mp = (p.M + 3) & ~3;
        const int items = kTileRows * (mp / 4);           // (row, column quad), item t = quad * 128 + row
        const int lo = items * split / p.splits, hi = items * (split + 1) / p.splits;
        for (int t = lo + (int)threadIdx.x; t < hi; t += kThreads) {
            float4 val[8];
#pragma unroll
            for (int s = 0; s < 8; ++s)
                val[s] = s < p.splits ? ld_dsmem_f4(sbase + (uint32_t)t * 16u, (uint32_t)s) : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                acc.x += val[s].x;
                acc.y += val[s].y;
                acc.z += val[s].z;
                acc.w += val[s].w;
            }
            const int r = t & (kTileRows - 1), q = t / kTileRows;
            const int n = tile * kTileRows + r;
            if (n < p.N) {
                const float o[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int m = 4 * q + c;
                    if (m < p.M) {
                        if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, o[c]);
                        else store_out<float>(p.y, (int64_t)m * p.N + n, o[c]);
                    }
                }
            }
        }
        // no CTA leaves while a peer may still read its shared memory
        cluster_sync_all();
        return;
    }

    // split K: the last CTA of this tile adds the partials in split order and
    // clears them
    if (p.splits > 1) {
        __shared__ unsigned int last;
        if (threadIdx.x == 0) {
            __threadfence();
            last = (atomicAdd(&p.counters[tile], 1u) == (unsigned)(p.splits - 1)) ? 1u : 0u;
        }
        __syncthreads();
        if (last) {
            __threadfence();
            const int rows = min(kTileRows, p.N - tile * kTileRows);
            const int mp = (p.M + 3) & ~3;
            const int quads = mp / 4;
            const int items = kTileRows * quads;      // (row, 4 columns); rows past N are skipped at the store
            // each thread owns up to kReduceItems (row, quad) items
            float4 acc[kReduceItems];
#pragma unroll
            for (int e = 0; e < kReduceItems; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            // up to four splits' loads in flight at once, added in split order
            for (int s0 = 0; s0 < p.splits; s0 += 4) {
                float4 val[4][kReduceItems];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4* src = reinterpret_cast<const float4*>(
                        p.partials + (size_t)((s0 + u) * p.tiles + tile) * kTileRows * (size_t)mp);
#pragma unroll
                    for (int e = 0; e < kReduceItems; ++e) {
                        const int t = (int)threadIdx.x + e * kThreads;   // t = quad * 128 + row
                        const int r = t & (kTileRows - 1), q = t / kTileRows;
                        val[u][e] = (s0 + u < p.splits && t < items) ? __ldcg(src + (size_t)r * quads + q)
                                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                // every call leaves the workspace all zero, so that any later
                // call (a stream-K plan reads it as tagged words) finds it clean
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float4* dst = reinterpret_cast<float4*>(
                        p.partials + (size_t)((s0 + u) * p.tiles + tile) * kTileRows * (size_t)mp);
#pragma unroll
                    for (int e = 0; e < kReduceItems; ++e) {
                        const int t = (int)threadIdx.x + e * kThreads;
                        const int r = t & (kTileRows - 1), q = t / kTileRows;
                        if (s0 + u < p.splits && t < items) __stcg(dst + (size_t)r * quads + q, make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int e = 0; e < kReduceItems; ++e) {
                        acc[e].x += val[u][e].x;
                        acc[e].y += val[u][e].y;
                        acc[e].z += val[u][e].z;
                        acc[e].w += val[u][e].w;
                    }
            }
#pragma unroll
            for (int e = 0; e < kReduceItems; ++e) {
                const int t = (int)threadIdx.x + e * kThreads;
                const int r = t & (kTileRows - 1), q = t / kTileRows;
                if (t < items && r < rows) {
                    const int n = tile * kTileRows + r;
                    const float o[4] = {acc[e].x, acc[e].y, acc[e].z, acc[e].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int m = 4 * q + c;
                        if (m < p.M) {
                            if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, o[c]);
                            else store_out<float>(p.y, (int64_t)m * p.N + n, o[c]);
                        }
                    }
                }
            }
            if (threadIdx.x == 0) p.counters[tile] = 0u;
        }
    }
}

}  // namespace

// Shared memory of the tensor-core kernel for MMA width nt; at least 116 KB so
// that a single CTA fits per SM (its 512 TMEM columns are then always free).
size_t qmm_tc_smem_bytes(int nt) {
    const size_t stage = (size_t)kRawStageBytes + (size_t)nt * kGroupK * 2;
    const size_t need = kStages * stage + 8 * kBarriers + 16;
    return need < 116 * 1024 ? 116 * 1024 : need;
}

int qmm_tc_tile_rows() { return kTileRows; }
int qmm_tc_group_k() { return kGroupK; }

cudaError_t launch_qmm_tc(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x, void* y, int y_bf16, float* partials,
                          unsigned int* counters, unsigned long long* share, unsigned int* fault, int M, int N, int K,
                          int splits, int cluster, int streamk_ctas, cudaStream_t stream) {
    QmmParams p;
    p.tmap_w = tmap_w;
    p.tmap_x = tmap_x;
    p.y = y;
    p.partials = partials;
    p.counters = counters;
    p.share = share;
    p.fault = fault;
    p.M = M;
    p.N = N;
    p.K = K;
    p.NT = (M + 15) / 16 * 16;
    p.groups = K / kGroupK;
    p.splits = splits;
    p.tiles = (N + kTileRows - 1) / kTileRows;
    p.y_bf16 = y_bf16;
    p.cluster = cluster;
    p.streamk = streamk_ctas > 0 ? 1 : 0;
    p.ctas = streamk_ctas;
    p.units = p.tiles * p.groups;
    if (p.streamk) p.splits = 1;
    const size_t smem = qmm_tc_smem_bytes(p.NT);
    static thread_local int prepared_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (prepared_device != dev) {
        for (auto k : {qmm_q4_0_tc_kernel<false>, qmm_q4_0_tc_kernel<true>}) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)qmm_tc_smem_bytes(32));
            if (e != cudaSuccess) return e;
        }
        prepared_device = dev;
    }
    // programmatic dependent launch: the prologue and the first weight copies
    // overlap the preceding kernel's tail
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(p.streamk ? streamk_ctas : p.tiles * splits));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (cluster && !p.streamk) ? 2 : 1;
    return p.streamk ? cudaLaunchKernelEx(&cfg, qmm_q4_0_tc_kernel<true>, p)
                     : cudaLaunchKernelEx(&cfg, qmm_q4_0_tc_kernel<false>, p);
}

// Clusters of `cluster` CTAs (MMA width nt) that the device holds at once; 0
// when such a launch is not possible.
int qmm_tc_max_active_clusters(int nt, int cluster) {
    if (cudaFuncSetAttribute(qmm_q4_0_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)qmm_tc_smem_bytes(32)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = qmm_tc_smem_bytes(nt);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, qmm_q4_0_tc_kernel<false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace qbw
