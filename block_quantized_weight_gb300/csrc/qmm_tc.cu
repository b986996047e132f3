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
// Warp roles: warps 0..15 dequantize (warp w: TMEM lanes 32 (w % 4) .. +31,
// block pair w / 4 of each K-group); warp 16 lane 0 issues the TMA copies;
// warp 17 lane 0 issues the MMAs.  Warps 0..3 also read the accumulator back.
//
// Dequantization, per weight pair: the code sits at bit 8, 12 or 16 of a word
// (shifted there if needed), is OR-ed with the exponent of 2^15, 2^11 or 2^7
// (giving 2^E + code exactly), and fma(f, d, -(2^E + 8) d) yields exactly
// d (code - 8): (2^E + 8) d needs at most 24 significant bits for E <= 15.
// The only rounding is the final conversion of the weight to bf16.
//
// Split K: each CTA writes its 128 x M partial tile to the workspace; the last
// CTA of a tile (counted with an atomic) adds the partials in split order and
// writes Y, then resets the counter so the workspace stays zero-filled.
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"

namespace qbw {
namespace {

constexpr int kTileRows = 128;
constexpr int kGroupK = 256;                  // K per pipeline stage (8 Q4_0 blocks)
constexpr int kGroupBytes = 144;              // raw bytes per row per K-group
constexpr int kDequantWarps = 16;
constexpr int kThreads = (kDequantWarps + 2) * 32;
constexpr int kStages = 4;                    // shared-memory stages (raw W + X)
constexpr int kAStages = 2;                   // TMEM A stages
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColsPerStage = kGroupK / 2;          // 2 bf16 per 32-bit column
constexpr uint32_t kDCol = kAStages * kAColsPerStage;     // accumulator columns start
constexpr uint32_t kRawStageBytes = kTileRows * kGroupBytes;   // 18432

// smem descriptor of a K-major, 128-byte-swizzled bf16 tile (8-row groups
// 1024 bytes apart), tcgen05 format.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1u << 16;                          // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                          // descriptor version (sm_100 family)
    d |= (uint64_t)2u << 61;                          // layout: 128-byte swizzle
    return d;
}

// instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4)                       // D format f32
           | (1u << 7)                     // A format bf16
           | (1u << 10)                    // B format bf16
           | ((uint32_t)(n >> 3) << 17)    // N / 8
           | ((uint32_t)(m >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 32 columns of this thread's TMEM lane <- v[0..31]
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// v[0..15] <- 16 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// f = (v & mask) | magic for one code each, then fma with the pair (d, d) and
// the pair constant k: exactly d (code - 8) per lane.
template <uint32_t ML, uint32_t MH>
__device__ __forceinline__ uint64_t wpair(uint32_t a, uint32_t b, uint32_t gl, uint32_t gh, uint64_t dd,
                                          uint64_t k) {
    uint64_t r;
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 t;\n\t"
        "lop3.b32 lo, %1, %6, %3, 0xEA;\n\t"
        "lop3.b32 hi, %2, %7, %4, 0xEA;\n\t"
        "mov.b64 t, {lo, hi};\n\t"
        "fma.rn.f32x2 %0, t, %5, %8;\n\t}"
        : "=l"(r)
        : "r"(a), "r"(b), "r"(gl), "r"(gh), "l"(dd), "n"(ML), "n"(MH), "l"(k));
    return r;
}

// bf16x2 of a fp32 pair: low half = first lane, high half = second lane
__device__ __forceinline__ uint32_t to_bf16x2(uint64_t p) {
    const float2 f = unpack2f(p);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}

// One Q4_0 block: scale d (fp16 bits) and qs words q0..q3 (qs bytes 4t..4t+3
// in word t).  Writes the 16 bf16x2 columns of the block's 32 weights in K
// order: column t' holds elements 2t' (low) and 2t'+1 (high).
__device__ __forceinline__ void dequant_block(uint32_t dbits, uint32_t q0, uint32_t q1, uint32_t q2, uint32_t q3,
                                              uint32_t* col) {
    const float d = half_bits_to_float(dbits);
    const uint32_t m15 = 0x47000000u, m11 = 0x45000000u, m7 = 0x43000000u;
    const float k15 = -32776.0f * d, k11 = -2056.0f * d, k7 = -136.0f * d;   // exact: <= 24 bits
    const uint64_t dd = pack2f(d, d);
    const uint64_t k15_15 = pack2f(k15, k15), k7_11 = pack2f(k7, k11), k11_11 = pack2f(k11, k11),
                   k15_7 = pack2f(k15, k7);
    const uint32_t q[4] = {q0, q1, q2, q3};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        // word q[t] = qs bytes 4t..4t+3; nibble n_i at bits 4i:
        //   n0 = elem 4t (lo of byte 0), n1 = elem 16+4t, n2 = elem 4t+1, n3 = elem 17+4t,
        //   n4 = elem 4t+2, n5 = elem 18+4t, n6 = elem 4t+3, n7 = elem 19+4t
        const uint32_t v = q[t];
        const uint32_t lft = v << 8;          // n0 at bit 8, n1 at bit 12
        const uint32_t rgt = v >> 12;         // n5 at bit 8, n6 at bit 12, n7 at bit 16
        // (elem 4t, 4t+1) = (n0 @8 of lft, n2 @8 of v)
        col[2 * t] = to_bf16x2(wpair<0x00000F00u, 0x00000F00u>(lft, v, m15, m15, dd, k15_15));
        // (elem 4t+2, 4t+3) = (n4 @16 of v, n6 @12 of rgt)
        col[2 * t + 1] = to_bf16x2(wpair<0x000F0000u, 0x0000F000u>(v, rgt, m7, m11, dd, k7_11));
        // (elem 16+4t, 17+4t) = (n1 @12 of lft, n3 @12 of v)
        col[8 + 2 * t] = to_bf16x2(wpair<0x0000F000u, 0x0000F000u>(lft, v, m11, m11, dd, k11_11));
        // (elem 18+4t, 19+4t) = (n5 @8 of rgt, n7 @16 of rgt)
        col[8 + 2 * t + 1] = to_bf16x2(wpair<0x00000F00u, 0x000F0000u>(rgt, rgt, m15, m7, dd, k15_7));
    }
}

struct QmmParams {
    CUtensorMap tmap_w;     // Q4_0 rows as 8-byte words, box (18, 128)
    CUtensorMap tmap_x;     // X [M][K] bf16, box (64, NT), 128-byte swizzle
    void* y;
    float* partials;        // [splits][M][N] fp32 (splits > 1)
    unsigned int* counters; // [tiles] (splits > 1)
    unsigned int* fault;
    int32_t M, N, K;
    int32_t NT;             // MMA N: M rounded up to 16
    int32_t groups;         // K / 256
    int32_t splits;
    int32_t y_bf16;
};

__global__ void __launch_bounds__(kThreads, 1) qmm_q4_0_tc_kernel(const __grid_constant__ QmmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / p.splits, split = blockIdx.x - tile * p.splits;
    const int g_begin = (int)((int64_t)p.groups * split / p.splits);
    const int g_end = (int)((int64_t)p.groups * (split + 1) / p.splits);
    const int ng = g_end - g_begin;

    // shared memory: [stages][raw W 18432 B | X NT x 256 bf16] (1024-aligned), barriers, TMEM slot
    const uint32_t xbytes = (uint32_t)p.NT * kGroupK * 2;            // 4 swizzle atoms of NT x 128 B
    const uint32_t stage_bytes = kRawStageBytes + xbytes;            // multiple of 1024
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kStages * stage_bytes;
    // barriers: full[kStages], empty[kStages], afull[kAStages], aempty[kAStages], dfull
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(kStages + s); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (uint32_t)(2 * kStages + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (uint32_t)(2 * kStages + kAStages + a); };
    const uint32_t dfull_bar = bar0 + 8u * (uint32_t)(2 * kStages + 2 * kAStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kStages * stage_bytes + 8 * (2 * kStages + 2 * kAStages + 1));

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kDequantWarps + 1);
        }
        for (int a = 0; a < kAStages; ++a) {
            mbar_init(afull_bar(a), kDequantWarps);
            mbar_init(aempty_bar(a), 1);
        }
        mbar_init(dfull_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "n"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == kDequantWarps) {
        // ---------------- producer: raw W and X tiles by TMA
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            prefetch_tmap(&p.tmap_w);
            prefetch_tmap(&p.tmap_x);
            for (int i = 0; i < ng && ok; ++i) {
                const int s = i % kStages;
                if (i >= kStages)
                    ok = mbar_wait_bounded(empty_bar(s), (uint32_t)((i / kStages) - 1) & 1u, p.fault,
                                           kFaultBulkWaitTimeout);
                if (!ok) break;
                const int g = g_begin + i;
                const uint32_t st = sbase + (uint32_t)s * stage_bytes;
                mbar_arrive_expect_tx(full_bar(s), kRawStageBytes + xbytes);
                tma_load_2d(st, &p.tmap_w, g * (kGroupBytes / 8), tile * kTileRows, full_bar(s), pol_w);
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    tma_load_2d(st + kRawStageBytes + (uint32_t)a * (uint32_t)p.NT * 128u, &p.tmap_x,
                                g * kGroupK + a * 64, 0, full_bar(s), 0ull);
            }
        }
    } else if (warp == kDequantWarps + 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kTileRows, p.NT);
            for (int i = 0; i < ng && ok; ++i) {
                const int s = i % kStages, a = i % kAStages;
                ok = mbar_wait_bounded(full_bar(s), (uint32_t)(i / kStages) & 1u, p.fault, kFaultMmaWaitTimeout) &&
                     mbar_wait_bounded(afull_bar(a), (uint32_t)(i / kAStages) & 1u, p.fault, kFaultMmaWaitTimeout);
                if (!ok) break;
                tc_fence_after();
                const uint32_t xs = sbase + (uint32_t)s * stage_bytes + kRawStageBytes;
#pragma unroll
                for (int k = 0; k < kGroupK / 16; ++k) {
                    const uint32_t a_tmem = tmem + (uint32_t)a * kAColsPerStage + (uint32_t)k * 8u;
                    const uint64_t bdesc = sw128_desc(xs + (uint32_t)(k >> 2) * (uint32_t)p.NT * 128u +
                                                      (uint32_t)(k & 3) * 32u);
                    tc_mma(tmem + kDCol, a_tmem, bdesc, idesc, (i > 0 || k > 0) ? 1u : 0u);
                }
                tc_commit(empty_bar(s));     // X tile of stage s consumed
                tc_commit(aempty_bar(a));    // TMEM A stage a consumed
            }
            // completes when every MMA issued above has finished, even after a
            // timeout (the accumulator is then not read, only TMEM released)
            tc_commit(dfull_bar);
        }
    } else {
        // ---------------- dequantizing warps
        const int quarter = warp & 3;                 // TMEM lanes 32 quarter .. +31
        const int pair = warp >> 2;                   // block pair of each K-group
        const int row = quarter * 32 + lane;          // weight row within the tile
        for (int i = 0; i < ng && ok; ++i) {
            const int s = i % kStages, a = i % kAStages;
            const bool got_w = mbar_wait_bounded(full_bar(s), (uint32_t)(i / kStages) & 1u, p.fault,
                                                 kFaultBulkWaitTimeout);
            const bool got_a = (i < kAStages) ||
                               mbar_wait_bounded(aempty_bar(a), (uint32_t)((i / kAStages) - 1) & 1u, p.fault,
                                                 kFaultMmaWaitTimeout);
            if (!__all_sync(0xffffffffu, got_w && got_a)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the pair's 36 bytes: V0 = [dA, qsA0, qsA1], V1..V3, V4 = [qsA14, qsA15, dB], V5..V8
            const uint32_t src = sbase + (uint32_t)s * stage_bytes + (uint32_t)row * kGroupBytes + (uint32_t)pair * 36u;
            uint32_t v[9];
#pragma unroll
            for (int w = 0; w < 9; ++w) v[w] = lds32(src + 4u * (uint32_t)w);
            uint32_t col[32];
            // block A: d = V0 lo; qs words (bytes 2..17 of the pair) realigned by 16 bits
            dequant_block(v[0] & 0xFFFFu, __funnelshift_r(v[0], v[1], 16), __funnelshift_r(v[1], v[2], 16),
                          __funnelshift_r(v[2], v[3], 16), __funnelshift_r(v[3], v[4], 16), col);
            // block B: d = V4 hi; qs words V5..V8
            dequant_block(v[4] >> 16, v[5], v[6], v[7], v[8], col + 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));     // raw W of stage s read
            tmem_st32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)a * kAColsPerStage + (uint32_t)pair * 32u,
                      col);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull_bar(a));
        }
        // ---------------- epilogue: warps 0..3 read D (128 rows x NT) and emit
        if (warp < 4) {
            const bool got = ok && mbar_wait_bounded(dfull_bar, 0u, p.fault, kFaultMmaWaitTimeout);
            if (__all_sync(0xffffffffu, got)) {
                tc_fence_after();
                const int n = tile * kTileRows + row;
                float* part = p.partials + (size_t)split * p.M * p.N;
                for (int c0 = 0; c0 < p.NT; c0 += 16) {
                    uint32_t dv[16];
                    tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + kDCol + (uint32_t)c0, dv);
                    tmem_wait_ld();
                    if (n < p.N) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = c0 + j;
                            if (m < p.M) {
                                const float val = __uint_as_float(dv[j]);
                                if (p.splits == 1) {
                                    if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, val);
                                    else store_out<float>(p.y, (int64_t)m * p.N + n, val);
                                } else {
                                    part[(size_t)m * p.N + n] = val;
                                }
                            }
                        }
                    }
                }
                __threadfence();              // partials visible before the split counter moves
            } else {
                ok = false;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        // no MMA may still be writing TMEM when it is released
        mbar_wait_bounded(dfull_bar, 0u, p.fault, kFaultMmaWaitTimeout);
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
    }

    // split K: the last CTA of this tile adds the partials in split order
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
            for (int t = threadIdx.x; t < rows * p.M; t += blockDim.x) {
                const int m = t / rows, r = t - m * rows;
                const int n = tile * kTileRows + r;
                float sum = 0.f;
                for (int s = 0; s < p.splits; ++s)
                    sum += __ldcg(p.partials + (size_t)s * p.M * p.N + (size_t)m * p.N + n);
                if (p.y_bf16) store_out<__nv_bfloat16>(p.y, (int64_t)m * p.N + n, sum);
                else store_out<float>(p.y, (int64_t)m * p.N + n, sum);
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
    const size_t need = kStages * stage + 8 * (2 * kStages + 2 * kAStages + 1) + 16;
    return need < 116 * 1024 ? 116 * 1024 : need;
}

int qmm_tc_tile_rows() { return kTileRows; }
int qmm_tc_group_k() { return kGroupK; }

cudaError_t launch_qmm_tc(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x, void* y, int y_bf16, float* partials,
                          unsigned int* counters, unsigned int* fault, int M, int N, int K, int splits,
                          cudaStream_t stream) {
    QmmParams p;
    p.tmap_w = tmap_w;
    p.tmap_x = tmap_x;
    p.y = y;
    p.partials = partials;
    p.counters = counters;
    p.fault = fault;
    p.M = M;
    p.N = N;
    p.K = K;
    p.NT = (M + 15) / 16 * 16;
    p.groups = K / kGroupK;
    p.splits = splits;
    p.y_bf16 = y_bf16;
    const size_t smem = qmm_tc_smem_bytes(p.NT);
    static thread_local int prepared_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (prepared_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(qmm_q4_0_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)qmm_tc_smem_bytes(32));
        if (e != cudaSuccess) return e;
        prepared_device = dev;
    }
    const int tiles = (N + kTileRows - 1) / kTileRows;
    qmm_q4_0_tc_kernel<<<tiles * splits, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace qbw
