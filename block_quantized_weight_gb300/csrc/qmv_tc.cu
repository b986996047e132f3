// qmv_tc.cu -- the M = 1 (and two-token) Q4_0 matrix-vector product y = W x,
// the fused Q4_0 gate+up, the Q4_K product and the mixed-bit (int2, int4,
// int8; groups of 32) products, on the fifth-generation tensor cores
// (tcgen05), for K a multiple of 256.  A Q4_K super-block (256 weights,
// 144 bytes) is exactly one unit's row segment; its codes enter A exactly
// (0..15), and the read-back applies d sc_j to each sub-block's dot product
// and subtracts dmin m_j times the sub-block's activation sum (the algebraic
// split of jouleclaw-loader-gguf BENCHMARKS, Q4_K NEON kernel).
//
// Why tensor cores for one token: on CUDA cores every weight costs a code
// extraction, an exact conversion to fp32 and a multiply-add, about 2.1
// instructions, and that instruction stream, not HBM, bounds the CUDA-core
// kernel.  On the tensor core the products and sums leave the decode warps,
// which only turn codes into an exact operand.
//
// Exact block scales.  A holds exact integer codes; the scale d of each block
// is applied after the MMA, in fp32, so no weight is rounded.  The MMA's N
// dimension carries one column pair per block instead of one per token: for a
// K-group of 256 (8 blocks), B is 16 columns where columns 2j and 2j + 1 hold
// two pieces of block j's activations (zeros elsewhere), and the row's thread
// adds d_j (D[2j] + D[2j + 1]) for j = 0..7, in that order.  Two forms
// (qmv_tc_common.cuh):
// * 8-bit (kind::f8f6f4, one token): Q4_0's c - 8 as two e4m3 operands,
//   c & 7 and 8 [bit 3 clear] (both 0 where c = 8), about 5.5 instructions
//   per 8 codes; Q4_K's codes 0..15 as one.  Activations are e4m3 pieces under
//   a power-of-two scale per block: two for bf16 x (exact), three for fp32
//   (about 12 bits; the third in a second B, one more MMA per K-step).  The
//   pieces and factors come from a table each CTA builds once.
// * bf16-code (kind::f16): c - 8 exact in bf16 (byte permute, LOP3 with the
//   exponent of 128, a packed add of -136), x as x_hi = bf16(x) and x_lo =
//   bf16(x - x_hi), 2^-17 relative; two bf16 tokens take those two columns.
//   It serves two tokens and shapes whose table would not fit.
//
// Work split (stream-K): the units are (128-row tile, K-group, matrix) triples
// in that order (one matrix, or gate then up); CTA c of C takes units
// [c U / C, (c + 1) U / C).  A tile
// that a CTA covers in full is written to y by that CTA.  A tile split between
// CTAs is finished by the CTA that covers its first unit (it reaches the tile
// last, at the end of its range).  Every other CTA on the tile starts its range
// inside it, completes its share early and publishes it then: one 64-bit word
// per row, (value, the launch's tag), in a scratch slot chosen from the grid
// id.  The finisher waits for words with its own tag (bounded), adds them
// after its own share in CTA order, writes y and marks them consumed (tag 0).
// Results are therefore bit-reproducible.
//
// Warp roles (16 warps): warps 0..11 are three sets of four dequantizing
// warps; set s takes the CTA's units s, s + 3, ...; warp 4s + q owns rows
// 32q .. 32q + 31 (its TMEM lane quarter) and one eighth of the group's B
// operand (lanes 0..7; the bf16-code Q4_K form: lanes 8q .. 8q + 7, while
// every lane loads activations for the sub-block sums).  Warp 12 lane 0
// issues the TMA copies of the raw rows (128 rows x 144 bytes per unit) into a
// 6-stage ring.  Warp 13 + s lane 0 issues set s's MMAs (M = 128, N = 16; 16
// K-steps per unit, 8 for 8-bit Q4_K) into one of set s's two D buffers.
// Each set's rows read D back one unit later, while the next unit's codes are
// already decoded in registers.
#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "qbw_device.cuh"
#include "qbw_internal.h"
#include "tc_common.cuh"
#include "qmv_tc_common.cuh"

namespace qbw {

// Split-tile scratch: each CTA's published share of its first tile, per row,
// as (fp32 bits, tag) with tag = the publishing launch's launch_tag() and 0 =
// consumed (all zero at load).  A launch uses slot (grid id mod kQtcSlots),
// chosen on the device, so launches close together in launch order (the
// launches of a captured graph, calls on several streams) take different
// slots, and a word is accepted only with the finisher's own launch tag: a
// stale word (left by a launch that faulted) or another launch's is never
// added.  Two launches kQtcSlots apart in launch order that run at the same
// time share a slot; the finisher then waits in vain and reports fault 4
// instead of adding a foreign value.
constexpr int kQtcSlots = 32;
constexpr int kQtcMaxCtas = 160;
constexpr int kQtcMaxTiles = 4096;
__device__ unsigned long long g_qtc_share[kQtcSlots][kQtcMaxCtas][2][128];

namespace {

using namespace qtc;

// NMAT = 1: y = W x.  NMAT = 2: out = gelu_tanh(Wg x) * (Wu x); the units of a
// (tile, group) are its gate and up halves, in that order (measured faster
// than all gate groups of a tile before its up groups, by about 1 %).  NTOK = 2 (with
// NMAT = 1 and bf16 activations): Y[m] = W X[m] for two token rows, which take
// the two B columns of each block that x_hi and x_lo take for one token.
// Each row keeps NCH = NMAT * NTOK sums (channels).  F8: the 8-bit form of
// the operands (Q4_0, one token; see codes_pair_e4m3), with F8 e4m3 pieces
// per activation: 2 for bf16 x, 3 for fp32 x (the third pieces in a second B,
// one more MMA per K-step on the same A, into the D column of the second
// piece).  F8 = 0: the bf16-code form.
template <int FMT, int NMAT, int NTOK, int F8>
__device__ __forceinline__ void qmv_tc_body(const QtcParams& p) {
    constexpr int NCH = NMAT * NTOK;
    static_assert(NCH <= 2, "at most two sums per row");
    static_assert(FMT == kFmtQ4 || (NMAT == 1 && NTOK == 1), "Q4_K: one matrix, one token");
    static_assert(F8 == 0 || ((F8 == 2 || F8 == 3) && NTOK == 1), "8-bit form: one token");
    // the int4-affine (MIX4) and int2-symmetric (MIX2) mixed-bit matrices:
    // 8-bit form with bf16 activations only (their scales and biases take the
    // B2 region)
    constexpr bool MIX4 = FMT == kFmtMix4, MIX2 = FMT == kFmtMix2, MIX = MIX4 || MIX2;
    // the int8 mixed-bit matrices: the two-operand 8-bit form (q = l + 16 h),
    // bf16 activations; a unit's 256 code bytes per row take two ring stages of
    // 128 bytes each, both with the unit's scales
    constexpr bool MIX8 = FMT == kFmtMix8;
    static_assert(!(MIX || MIX8) || F8 == 2 || F8 == 3, "mixed-bit forms: the 8-bit form");
    // where a mixed-bit form's scales (and biases) come from: copied with the
    // codes for groups of 32 (int2 and int4 into the B2 region, which the
    // fp32 form needs for its third pieces, so only with bf16 x; int8 into
    // its ring stages); otherwise read by the threads from global memory
    const bool mix_sc_copied = !(MIX || MIX8) || (p.mgshift == 5 && (F8 == 2 || MIX8));
    // the 8-bit form of Q4_K: one A operand (codes 0..15), 8 K-steps per unit
    constexpr bool Q4K8 = F8 != 0 && FMT == kFmtQ4K;
    // one A operand of codes (Q4_K's 0..15, the int4 and int2 mixed-bit forms)
    constexpr bool ONE_OP = Q4K8 || MIX;
    constexpr int kSteps = ONE_OP ? 8 : 16;
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
    if (threadIdx.x == 0) *reinterpret_cast<uint32_t*>(smem + kOffXflag) = 0u;     // set by the table build
    const uint64_t gid = grid_id();
    const uint32_t tag = launch_tag();
    unsigned long long* share = &g_qtc_share[gid % kQtcSlots][0][0][0];   // [cta][matrix][row]

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    float* part = reinterpret_cast<float*>(smem + kOffPart);      // [set][local tile][matrix][row]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
    bool ok = true;

    // zero B operands (only their fixed activation positions are ever written
    // again) and the per-set partial rows
    // (B2 too, except where it is the int2 / int4 forms' scale ring, which the
    // copies below start filling at once; the fp32 forms' third pieces need it
    // zero like B)
    for (int i = threadIdx.x; i < (int)((MIX && mix_sc_copied ? 1 : 2) * kSets * kBBytes / 16); i += kThreads)
        sts128(sbase + kOffB + 16u * (uint32_t)i, make_uint4(0u, 0u, 0u, 0u));
    for (int i = threadIdx.x; i < kSets * kMaxLocalTiles * 2 * kTileRows; i += kThreads) part[i] = 0.f;
    for (int i = threadIdx.x; i < kProducerWarp * 32 * 3; i += kThreads)       // acc_q and fixups
        reinterpret_cast<uint32_t*>(smem + kOffQ)[i] = 0u;

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
            if (NMAT == 2 || ((MIX || MIX8) && mix_sc_copied)) prefetch_tmap(&p.tmap_w[1]);
            if (MIX4 && mix_sc_copied) prefetch_tmap(&p.tmap_bi);
            // weights do not depend on the preceding grid: start streaming now
            const bool sc_tma = mix_sc_copied;
            if constexpr (MIX8) {
                // unit i's halves in ring stages (2i) % 6 and (2i + 1) % 6: codes
                // (16 words of a row), then the unit's scales (2 words)
                for (int i = 0; i < n && ok; ++i) {
                    const int u = u0 + i, t = u / G, g = u - t * G;
                    for (int hs = 0; hs < 2; ++hs) {
                        const int q = 2 * i + hs, s = q % kStages;
                        if (q >= kStages)
                            ok = mbar_wait_bounded(empty_bar(bar0, s), (uint32_t)((q / kStages) - 1) & 1u, p.fault,
                                                   kFaultBulkWaitTimeout);
                        if (!ok) break;
                        const uint32_t dst = sbase + (uint32_t)s * kRawStageBytes;
                        mbar_arrive_expect_tx(full_bar(bar0, s), sc_tma ? kMix8StageBytes : kMixCodeBytes);
                        tma_load_2d(dst, &p.tmap_w[0], g * 32 + 16 * hs, t * kTileRows, full_bar(bar0, s),
                                    policy_evict_first());
                        if (sc_tma)
                            tma_load_2d(dst + kMixCodeBytes, &p.tmap_w[1], g * 2, t * kTileRows, full_bar(bar0, s),
                                        policy_evict_first());
                    }
                }
            }
            for (int i = 0; i < (MIX8 ? 0 : n) && ok; ++i) {
                const int s = i % kStages;
                if (i >= kStages)
                    ok = mbar_wait_bounded(empty_bar(bar0, s), (uint32_t)((i / kStages) - 1) & 1u, p.fault,
                                           kFaultBulkWaitTimeout);
                if (!ok) break;
                const int u = u0 + i, ug = u / NMAT, mat = u - ug * NMAT, t = ug / G, g = ug - t * G;
                if constexpr (MIX) {
                    // codes (16 or 8 words of a row), then scales and biases (2 words each)
                    const uint32_t sdst = sbase + kOffB2 + (uint32_t)s * kMixScaleBytes;
                    const uint32_t code_bytes = kTileRows * (MIX4 ? 128u : 64u);
                    mbar_arrive_expect_tx(full_bar(bar0, s), sc_tma ? (MIX4 ? kMixStageBytes : kMix2StageBytes)
                                                                    : code_bytes);
                    tma_load_2d(sbase + (uint32_t)s * kRawStageBytes, &p.tmap_w[0], g * (MIX4 ? 16 : 8),
                                t * kTileRows, full_bar(bar0, s), policy_evict_first());
                    if (sc_tma) {
                        tma_load_2d(sdst, &p.tmap_w[1], g * 2, t * kTileRows, full_bar(bar0, s),
                                    policy_evict_first());
                        if constexpr (MIX4)
                            tma_load_2d(sdst + kMixScaleBytes / 2, &p.tmap_bi, g * 2, t * kTileRows,
                                        full_bar(bar0, s), policy_evict_first());
                    }
                } else {
                    mbar_arrive_expect_tx(full_bar(bar0, s), kRawStageBytes);
                    tma_load_2d(sbase + (uint32_t)s * kRawStageBytes, &p.tmap_w[mat], g * kGroupWords,
                                t * kTileRows, full_bar(bar0, s), policy_evict_first());
                }
            }
            // every copy of this launch is issued: warm L2 with the first units
            // (a ring's worth) that this CTA index loads in the next launch
            if (ok && p.next_units > 0 && cta < p.next_ctas) {
                const int v0 = unit_begin(cta, p.next_units, p.next_ctas);
                const int v1 = unit_begin(cta + 1, p.next_units, p.next_ctas);
                for (int i = 0; i < kStages && v0 + i < v1; ++i) {
                    const int u = v0 + i, ug = u / p.next_nmat, mat = u - ug * p.next_nmat, t = ug / p.next_groups,
                              g = ug - t * p.next_groups;
                    tma_prefetch_2d(&p.next_tmap[mat], g * kGroupWords, t * kTileRows);
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
            const uint64_t b20 = sw128_desc(sbase + kOffB2 + (uint32_t)set * kBBytes);
            uint32_t phase = 0;
            for (int i = set; i < n; i += kSets) {
                // the set's k-th unit accumulates into D buffer k % 2
                const uint32_t d_tmem = tmem + kDCol + 32u * (uint32_t)set + 16u * phase;
                // K-steps 0..7 as soon as the first half is written, 8..15 after the second
                ok = mbar_wait_bounded(afull_bar(bar0, set, 0), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kSteps / 2; ++k) {
                    const uint64_t bo = (uint64_t)((k >> 2) * 128 + (k & 3) * 2);
                    if constexpr (F8) {
                        tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + bo, idesc, k > 0 ? 1u : 0u);
                        if constexpr (F8 == 3) tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b20 + bo, idesc, 1u);
                    } else {
                        tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + bo, idesc, k > 0 ? 1u : 0u);
                    }
                }
                tc_commit(aempty_bar(bar0, set, 0));
                ok = mbar_wait_bounded(afull_bar(bar0, set, 1), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int k = kSteps / 2; k < kSteps; ++k) {
                    const uint64_t bo = (uint64_t)((k >> 2) * 128 + (k & 3) * 2);
                    if constexpr (F8) {
                        tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + bo, idesc, 1u);
                        if constexpr (F8 == 3) tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b20 + bo, idesc, 1u);
                    } else {
                        tc_mma(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + bo, idesc, 1u);
                    }
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
        const uint32_t raw_row = (uint32_t)(32 * q + lane) * ((MIX4 || MIX8) ? 128u : (MIX2 ? 64u : 144u));
        const uint32_t bbuf = sbase + kOffB + (uint32_t)set * kBBytes;
        // The lane's 8-element slot xl of the group's activations: Q4_0, lanes
        // 0..7 load slots 8q .. 8q + 7 and write them into B; Q4_K, every lane
        // loads slot `lane` (the sub-block sums need all 256) and the lanes of
        // slots 8q .. 8q + 7 write them.  Slot xl is elements 8 xl .. 8 xl + 7 of
        // the group: swizzle atom xl / 8, block j = xl / 4, B rows 2j (x_hi)
        // and 2j + 1 (x_lo), in K-half xl / 16.
        // (the 8-bit form's B-writing lanes read their slot from the table)
        constexpr bool kAllLanesX = FMT == kFmtQ4K && !Q4K8;
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
        // 8-bit Q4_K: sub-block bj at K-step bj, rows 2bj (piece 0) and 2bj + 1
        const uint32_t kb = (uint32_t)((bj & 3) * 32 + 8 * (xl & 3));
        const uint32_t k8_p0 = bbuf + b_byte(bj >> 2, 2 * bj, kb), k8_p1 = bbuf + b_byte(bj >> 2, 2 * bj + 1, kb);
        const int bhalf = xl >> 4;
        const int row = 32 * q + lane;
        // 8-bit form: the activation table of the K-groups g of this CTA's
        // units, group g in slot (g - xg0) mod G, built by the twelve
        // dequantizing warps; the host launches this form only where the table
        // holds every group needed.
        const int xg0 = (u0 / NMAT) % G;
        if constexpr (F8) {
            const int cnt = n > 0 ? min(G, (u1 - 1) / NMAT - u0 / NMAT + 1) : 0;
            if (cnt > kXtGroups) record_fault(p.fault, kFaultPlan);
            // (with the groups' sums of x where a min or bias term takes them)
            build_x_table<false, F8, Q4K8 || MIX4, MIX8>(sbase, p.x, xg0, G, min(cnt, kXtGroups), warp, lane,
                                                         kProducerWarp);
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
                                   (unsigned long long)__float_as_uint(v) | ((unsigned long long)tag << 32));
                }
            }
            counted = true;
        };
        // The unit loop, in two compiled forms: kGuard (the 8-bit form, when
        // some group of this CTA's table is flagged) adds each flagged unit's
        // error-check term and the flagged segments' exact corrections; the
        // other form carries none of that code.
        auto run = [&](auto guard_tag) {
            constexpr bool kGuard = decltype(guard_tag)::value;
            // the row's sums of the tile being accumulated, one per matrix; in the
            // 8-bit form also the error-check terms of its flagged units
            float acc[NCH];
    #pragma unroll
            for (int m = 0; m < NCH; ++m) acc[m] = 0.f;
            float* acc_q = reinterpret_cast<float*>(smem + kOffQ) + 2 * threadIdx.x;
            uint32_t* fixups = reinterpret_cast<uint32_t*>(smem + kOffFix) + threadIdx.x;
            int acc_tile = -1, pend_tile = -1, pend_mat = 0;
            // 8-bit form: the exact sum of w r over this set's units of tile T,
            // matrix m (r: what the pieces miss), for a segment the check flags
            auto segment_correction = [&](int T, int m) -> float {
                const int64_t nrow = (int64_t)T * kTileRows + row;
                float corr = 0.f;
                if (nrow >= p.N) return corr;
                for (int i = set; i < n; i += kSets) {
                    const int u = u0 + i, ug = u / NMAT, mat = u - ug * NMAT, t = ug / G, g = ug - t * G;
                    if (t > T) break;
                    if (t < T || mat != m) continue;
                    int sl = g - xg0;
                    if (sl < 0) sl += G;
                    if (sl >= kXtGroups) sl = 0;
                    if (!group_flagged(sbase, sl)) continue;     // no residuals
                    if constexpr (MIX || MIX8) {
                        uint32_t s8[4];
                        mix_unit_values(p.msc + nrow * (p.K >> p.mgshift), g, p.mgshift, s8);
                        corr += unit_correction<FMT, F8, false>(
                            p.w[0] + nrow * p.row_bytes + (int64_t)g * (MIX8 ? 256 : (MIX4 ? 128 : 64)), p.x, g,
                            sbase, sl, make_uint4(s8[0], s8[1], s8[2], s8[3]));
                    }
                    else
                        corr += unit_correction<FMT, F8 ? F8 : 2, false>(
                            p.w[m] + nrow * p.row_bytes + (int64_t)g * 144, p.x, g, sbase, sl);
                }
                return corr;
            };
            // the set's partial rows of acc_tile -> part[]; in the 8-bit form a
            // segment that fails the error check (its units' terms, summed in
            // acc_q) gets bit 2 (acc_tile - tile0) + m in fixups, and its exact
            // correction is added after the unit loop
            auto flush = [&]() {
                if (acc_tile < 0) return;
    #pragma unroll
                for (int m = 0; m < NCH; ++m) {
                    if constexpr (kGuard) {
                        const float q = acc_q[m];
                        if (q != 0.f) {
                            acc_q[m] = 0.f;
                            if (segment_needs_correction(q)) *fixups |= 1u << (2 * (acc_tile - tile0) + m);
                        }
                    }
                    part[part_at(set, acc_tile - tile0, m, row)] = acc[m];
                }
            };
            auto add_unit = [&](float r0, float r1) {
                if (pend_tile != acc_tile) {
                    flush();
    #pragma unroll
                    for (int m = 0; m < NCH; ++m) acc[m] = 0.f;
                    acc_tile = pend_tile;
                    // a first-tile share that needs its correction is published
                    // after the unit loop instead
                    if (!counted && pend_tile > tile0 && !__any_sync(0xffffffffu, kGuard && (*fixups & 3u) != 0u))
                        count_in();
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
            [[maybe_unused]] uint32_t pend_bb[4] = {0u, 0u, 0u, 0u};     // the mixed-bit form's biases
            float pend_sx = 0.f;     // Q4_K: the previous unit's sub-block sum of this lane's group of 4
            int pend_sl = 0;         // 8-bit form: the previous unit's table slot
            // 8-bit form, a unit of a flagged group (the sign of its c_0; after
            // add_unit has moved acc_tile to it): its error-check term into the
            // segment's sum
            auto check_unit = [&](const uint32_t (&dv)[16], const float (&c)[8]) {
                float a[8];
                table_f8(sbase, kOffXr, pend_sl, a);
                acc_q[pend_mat] += unit_check_term<FMT>(dv, pend_dd, c, a);
            };
            int k = 0;
            for (int i = set; i < n; i += kSets, ++k) {
                const int u = u0 + i, ug = u / NMAT, mat = u - ug * NMAT, t = ug / G, g = ug - t * G;
                // the unit's ring stage and its completion parity (the int8 form:
                // its first half's stage; the second follows it)
                const int s = MIX8 ? (2 * i) % kStages : i % kStages;
                const uint32_t spar = (uint32_t)((MIX8 ? 2 * i : i) / kStages) & 1u;
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
                // the block scales (and int4 biases) of this unit and row; the
                // mixed-bit forms with groups larger than 32 read theirs from
                // global memory here, ahead of the stage wait (they are needed at
                // the read-back, one unit later)
                uint32_t dd[4];
                [[maybe_unused]] uint32_t bb[4];
                if constexpr (MIX || MIX8) {
                    if (!mix_sc_copied) {
    #pragma unroll
                        for (int P = 0; P < 4; ++P) dd[P] = bb[P] = 0u;
                        const int64_t nrow = (int64_t)t * kTileRows + row;
                        if (nrow < p.N) {
                            mix_unit_values(p.msc + nrow * (p.K >> p.mgshift), g, p.mgshift, dd);
                            if constexpr (MIX4) mix_unit_values(p.mbi + nrow * (p.K >> p.mgshift), g, p.mgshift, bb);
                        }
                    }
                }
                const bool got = mbar_wait_bounded(full_bar(bar0, s), spar, p.fault, kFaultBulkWaitTimeout);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint32_t src = sbase + (uint32_t)s * kRawStageBytes + raw_row;
                uint32_t v[36];
                if constexpr (MIX8) {
                    // the first half's 8 swizzled code chunks, then the unit's scales
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 w = lds128(src + (((uint32_t)j ^ (uint32_t)(row & 7)) << 4));
                        v[4 * j] = w.x;
                        v[4 * j + 1] = w.y;
                        v[4 * j + 2] = w.z;
                        v[4 * j + 3] = w.w;
                    }
                    if (mix_sc_copied) {
                        const uint4 sv =
                            lds128(sbase + (uint32_t)s * kRawStageBytes + kMixCodeBytes + (uint32_t)row * 16u);
                        dd[0] = sv.x;
                        dd[1] = sv.y;
                        dd[2] = sv.z;
                        dd[3] = sv.w;
                    }
                } else if constexpr (MIX) {
                    // the row's 8 (4) swizzled code chunks, then its scales (and biases)
    #pragma unroll
                    for (int j = 0; j < (MIX4 ? 8 : 4); ++j) {
                        const uint32_t sw = MIX4 ? (uint32_t)(row & 7) : (uint32_t)((row >> 1) & 3);
                        const uint4 w = lds128(src + (((uint32_t)j ^ sw) << 4));
                        v[4 * j] = w.x;
                        v[4 * j + 1] = w.y;
                        v[4 * j + 2] = w.z;
                        v[4 * j + 3] = w.w;
                    }
                    if (mix_sc_copied) {
                        const uint32_t ssrc = sbase + kOffB2 + (uint32_t)s * kMixScaleBytes + (uint32_t)row * 16u;
                        const uint4 sv = lds128(ssrc);
                        dd[0] = sv.x;
                        dd[1] = sv.y;
                        dd[2] = sv.z;
                        dd[3] = sv.w;
                        if constexpr (MIX4) {
                            const uint4 bv = lds128(ssrc + kMixScaleBytes / 2);
                            bb[0] = bv.x;
                            bb[1] = bv.y;
                            bb[2] = bv.z;
                            bb[3] = bv.w;
                        }
                    }
                } else {
    #pragma unroll
                    for (int j = 0; j < 9; ++j) {
                        const uint4 w = lds128(src + 16u * (uint32_t)j);
                        v[4 * j] = w.x;
                        v[4 * j + 1] = w.y;
                        v[4 * j + 2] = w.z;
                        v[4 * j + 3] = w.w;
                    }
    #pragma unroll
                    for (int P = 0; P < 4; ++P) dd[P] = (FMT == kFmtQ4K) ? v[P] : scale_pair(v, P);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(bar0, s));     // raw rows of stage s read
                uint32_t c0[32];
                [[maybe_unused]] uint32_t c1[32];     // not used by the one-operand Q4_K form
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
                // pieces of their slot
                int cur_sl = 0;
                uint2 bp0 = make_uint2(0u, 0u);
                [[maybe_unused]] uint2 bp1 = bp0, bp2 = bp0;     // the 8-bit forms' second and third pieces
                [[maybe_unused]] uint2 bq0 = bp0, bq1 = bp0, bq2 = bp0;     // the int8 form's pieces times 16
                if constexpr (F8) {
                    cur_sl = g - xg0;
                    if (cur_sl < 0) cur_sl += G;
                    if (cur_sl >= kXtGroups) cur_sl = 0;       // never: the host checks the table size
                    if (bwriter) {
                        const uint32_t ch = (uint32_t)(cur_sl * 32 + xl);
                        const uint4 tq = lds128(sbase + kOffXt + ch * 16u);
                        bp0 = make_uint2(tq.x, tq.y);
                        bp1 = make_uint2(tq.z, tq.w);
                        if constexpr (F8 == 3)
                            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                                         : "=r"(bp2.x), "=r"(bp2.y)
                                         : "r"(sbase + kOffXt2 + ch * 8u));
                        if constexpr (MIX) {     // the code words' order of weights
                            bp0 = perm_mix4(bp0);
                            bp1 = perm_mix4(bp1);
                            if constexpr (F8 == 3) bp2 = perm_mix4(bp2);
                        }
                        if constexpr (MIX8) {    // the second K-step's pieces: 16 x
                            bq0 = times16_e4m3(bp0);
                            bq1 = times16_e4m3(bp1);
                            if constexpr (F8 == 3) bq2 = times16_e4m3(bp2);
                        }
                    }
                }
                const uint32_t prev = (uint32_t)(k - 1) & 1u;     // completion parity of the previous unit
                // ---- half 0: K 0..127 (block pairs 0, 1; B atoms 0, 1 written by warps 0, 1)
                if constexpr (MIX4) codes_mix4_e4m3<0>(v, c0);
                else if constexpr (MIX2) codes_mix2_e4m3<0>(v, c0);
                else if constexpr (MIX8) codes_mix8_e4m3<0>(v, c0);
                else if constexpr (Q4K8) codes_q4k_e4m3<0>(v, c0);
                else if constexpr (F8) codes_pair_e4m3<0>(v, c0);
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
                    if constexpr (ONE_OP) {
                        sts64(k8_p0, bp0);
                        sts64(k8_p1, bp1);
                        if constexpr (F8 == 3) sts64(k8_p1 + (kOffB2 - kOffB), bp2);
                    } else if constexpr (F8) {
                        sts64(f8_p0, bp0);
                        sts64(f8_p1, bp1);
                        sts64(f8_n0, MIX8 ? bq0 : make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                        sts64(f8_n1, MIX8 ? bq1 : make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                        if constexpr (F8 == 3) {     // third pieces: B2, the second piece's rows
                            sts64(f8_p1 + (kOffB2 - kOffB), bp2);
                            sts64(f8_n1 + (kOffB2 - kOffB),
                                  MIX8 ? bq2 : make_uint2(bp2.x ^ 0x80808080u, bp2.y ^ 0x80808080u));
                        }
                    } else {
                        sts128(b_hi, bhi);
                        sts128(b_lo, blo);
                    }
                    fence_proxy_async_smem();     // B visible to the tensor core
                }
                tmem_st32(a_taddr, c0);
                if constexpr (!ONE_OP) {
                    if constexpr (MIX8) codes_mix8_e4m3<1>(v, c1);
                    else if constexpr (F8) codes_pair_e4m3<1>(v, c1);
                    else codes_pair<FMT, 1>(v, c1);
                    tmem_wait_st();
                    tmem_st32(a_taddr + 32u, c1);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(bar0, set, 0));
                // ---- half 1: K 128..255 (block pairs 2, 3; B atoms 2, 3 written by warps 2, 3)
                if constexpr (MIX8) {
                    // the second half's codes, in the unit's next ring stage
                    const int s1 = (2 * i + 1) % kStages;
                    const bool got1 = mbar_wait_bounded(full_bar(bar0, s1), (uint32_t)((2 * i + 1) / kStages) & 1u,
                                                        p.fault, kFaultBulkWaitTimeout);
                    if (!__all_sync(0xffffffffu, got1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t src1 = sbase + (uint32_t)s1 * kRawStageBytes + raw_row;
    #pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 w = lds128(src1 + (((uint32_t)j ^ (uint32_t)(row & 7)) << 4));
                        v[4 * j] = w.x;
                        v[4 * j + 1] = w.y;
                        v[4 * j + 2] = w.z;
                        v[4 * j + 3] = w.w;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(bar0, s1));
                }
                if constexpr (MIX4) codes_mix4_e4m3<1>(v, c0);
                else if constexpr (MIX2) codes_mix2_e4m3<1>(v, c0);
                else if constexpr (MIX8) codes_mix8_e4m3<0>(v, c0);
                else if constexpr (Q4K8) codes_q4k_e4m3<1>(v, c0);
                else if constexpr (F8) codes_pair_e4m3<2>(v, c0);
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
                    if constexpr (ONE_OP) {
                        sts64(k8_p0, bp0);
                        sts64(k8_p1, bp1);
                        if constexpr (F8 == 3) sts64(k8_p1 + (kOffB2 - kOffB), bp2);
                    } else if constexpr (F8) {
                        sts64(f8_p0, bp0);
                        sts64(f8_p1, bp1);
                        sts64(f8_n0, MIX8 ? bq0 : make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                        sts64(f8_n1, MIX8 ? bq1 : make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                        if constexpr (F8 == 3) {     // third pieces: B2, the second piece's rows
                            sts64(f8_p1 + (kOffB2 - kOffB), bp2);
                            sts64(f8_n1 + (kOffB2 - kOffB),
                                  MIX8 ? bq2 : make_uint2(bp2.x ^ 0x80808080u, bp2.y ^ 0x80808080u));
                        }
                    } else {
                        sts128(b_hi, bhi);
                        sts128(b_lo, blo);
                    }
                    fence_proxy_async_smem();
                }
                if constexpr (ONE_OP) {
                    tmem_st32(a_taddr + 32u, c0);
                } else {
                    tmem_st32(a_taddr + 64u, c0);
                    if constexpr (MIX8) codes_mix8_e4m3<1>(v, c1);
                    else if constexpr (F8) codes_pair_e4m3<3>(v, c1);
                    else codes_pair<FMT, 3>(v, c1);
                    tmem_wait_st();
                    tmem_st32(a_taddr + 96u, c1);
                }
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
                    if constexpr (MIX2) {
                        // sum_j (sc_j c_j) (D[2j] + D[2j + 1] / 16), as Q4_0's d_j
                        float c[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        r0 = unit_dot_e4m3(dv, pend_dd, c);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (MIX4) {
                        float c[8], sx[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        table_f8(sbase, kOffXs, pend_sl, sx);
                        r0 = unit_dot_mix4_e4m3(dv, pend_dd, pend_bb, c, sx);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (Q4K8) {
                        float c[8], sx[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        table_f8(sbase, kOffXs, pend_sl, sx);
                        r0 = unit_dot_q4k_e4m3(dv, pend_dd, c, sx);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (FMT == kFmtQ4K) {
                        r0 = unit_dot_q4k(dv, pend_dd, pend_sx);
                        add_unit(r0, r1);
                    } else if constexpr (F8) {
                        float c[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        r0 = unit_dot_e4m3(dv, pend_dd, c);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else {
                        unit_dot<NTOK>(dv, pend_dd, r0, r1);
                        add_unit(r0, r1);
                    }
                }
    #pragma unroll
                for (int P = 0; P < 4; ++P) {
                    pend_dd[P] = dd[P];
                    if constexpr (MIX4) pend_bb[P] = bb[P];
                }
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
                    if constexpr (MIX2) {
                        // sum_j (sc_j c_j) (D[2j] + D[2j + 1] / 16), as Q4_0's d_j
                        float c[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        r0 = unit_dot_e4m3(dv, pend_dd, c);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (MIX4) {
                        float c[8], sx[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        table_f8(sbase, kOffXs, pend_sl, sx);
                        r0 = unit_dot_mix4_e4m3(dv, pend_dd, pend_bb, c, sx);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (Q4K8) {
                        float c[8], sx[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        table_f8(sbase, kOffXs, pend_sl, sx);
                        r0 = unit_dot_q4k_e4m3(dv, pend_dd, c, sx);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else if constexpr (FMT == kFmtQ4K) {
                        r0 = unit_dot_q4k(dv, pend_dd, pend_sx);
                        add_unit(r0, r1);
                    } else if constexpr (F8) {
                        float c[8];
                        table_f8(sbase, kOffXc, pend_sl, c);
                        r0 = unit_dot_e4m3(dv, pend_dd, c);
                        add_unit(r0, r1);
                        if constexpr (kGuard)
                            if (__float_as_uint(c[0]) >> 31) check_unit(dv, c);
                    } else {
                        unit_dot<NTOK>(dv, pend_dd, r0, r1);
                        add_unit(r0, r1);
                    }
                }
            }
            flush();
            if constexpr (kGuard) {
                // the flagged segments' exact corrections (rare: activations whose
                // elements far below their block's largest carry the row's sum)
                uint32_t fx = *fixups;
                *fixups = 0u;
                while (fx != 0u) {
                    const int b = __ffs(fx) - 1;
                    fx &= fx - 1u;
                    part[part_at(set, b >> 1, b & 1, row)] += segment_correction(tile0 + (b >> 1), b & 1);
                }
            }
            if (!counted) count_in();
        };
        bool guard = false;
        if constexpr (F8 != 0) guard = lds32(sbase + kOffXflag) != 0u;
        if constexpr (F8 != 0) {
            if (guard) run(std::true_type{});
            else run(std::false_type{});
        } else {
            run(std::false_type{});
        }
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
                        const unsigned long long w = wait_tag_u64(src, tag, p.fault, kFaultShareWaitTimeout);
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
    qmv_tc_body<kFmtQ4, NMAT, NTOK, 0>(p);
}

// one token: the 8-bit operand form, XP pieces per activation (2: bf16, 3: fp32)
template <int NMAT, int XP>
__global__ void __launch_bounds__(kThreads, 1) qmv_q4_0_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4, NMAT, 1, XP>(p);
}

__global__ void __launch_bounds__(kThreads, 1) qmv_q4_k_tc_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4K, 1, 1, 0>(p);
}

// Q4_K in the 8-bit operand form, XP pieces per activation
template <int XP>
__global__ void __launch_bounds__(kThreads, 1) qmv_q4_k_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtQ4K, 1, 1, XP>(p);
}

// the int4-affine mixed-bit matrices (groups of 32) in the 8-bit operand
// form, bf16 activations
template <int XP>
__global__ void __launch_bounds__(kThreads, 1) qmv_mix4_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtMix4, 1, 1, XP>(p);
}

// the int2-symmetric mixed-bit matrices (groups of 32), likewise
template <int XP>
__global__ void __launch_bounds__(kThreads, 1) qmv_mix2_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtMix2, 1, 1, XP>(p);
}

// the int8 mixed-bit matrices (groups of 32), the two-operand 8-bit form
template <int XP>
__global__ void __launch_bounds__(kThreads, 1) qmv_mix8_tc_e4m3_kernel(const __grid_constant__ QtcParams p) {
    qmv_tc_body<kFmtMix8, 1, 1, XP>(p);
}

// Every kernel of this file may take kSmemBytes of dynamic shared memory (once
// per device and thread).
cudaError_t prepare_qtc_kernels() {
    static thread_local int prepared_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (prepared_device == dev) return cudaSuccess;
    for (auto f : {qmv_q4_0_tc_kernel<1, 1>, qmv_q4_0_tc_kernel<2, 1>, qmv_q4_0_tc_kernel<1, 2>,
                   qmv_q4_0_tc_e4m3_kernel<1, 2>, qmv_q4_0_tc_e4m3_kernel<2, 2>, qmv_q4_0_tc_e4m3_kernel<1, 3>,
                   qmv_q4_0_tc_e4m3_kernel<2, 3>, qmv_q4_k_tc_kernel, qmv_q4_k_tc_e4m3_kernel<2>,
                   qmv_q4_k_tc_e4m3_kernel<3>, qmv_mix4_tc_e4m3_kernel<2>, qmv_mix2_tc_e4m3_kernel<2>,
                   qmv_mix8_tc_e4m3_kernel<2>, qmv_mix4_tc_e4m3_kernel<3>, qmv_mix2_tc_e4m3_kernel<3>,
                   qmv_mix8_tc_e4m3_kernel<3>}) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    prepared_device = dev;
    return cudaSuccess;
}

cudaError_t launch_qtc(void (*kernel)(QtcParams), const QtcParams& p, int ctas, cudaStream_t stream) {
    cudaError_t e = prepare_qtc_kernels();
    if (e != cudaSuccess) return e;
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

// Whether the 8-bit form's activation table holds every K-group that a CTA's
// unit range needs (one token, nmat matrices; CTAs = min(units, SMs)).
bool table_fits(int nmat, int units, int groups, int sm_count) {
    const int ctas = units < sm_count ? units : sm_count;
    const int per_cta = (units + ctas - 1) / ctas;
    return std::min(groups, (per_cta - 1) / nmat + 2) <= kXtGroups;
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
cudaError_t launch_qmv_tc(int fmt, int nmat, int ntok, const CUtensorMap* tmap_w, const void* const* w,
                          const void* x, int x_bf16, void* y, int y_bf16, int N, int K, int sm_count,
                          unsigned int* fault, cudaStream_t stream, const QtcNextLaunch* next) {
    if (nmat * ntok > 2 || (ntok == 2 && !x_bf16)) return cudaErrorInvalidValue;
    if (fmt == kFmtQ4K && nmat * ntok != 1) return cudaErrorInvalidValue;
    QtcParams p;
    p.tmap_w[0] = tmap_w[0];
    p.tmap_w[1] = tmap_w[nmat == 2 ? 1 : 0];
    p.w[0] = static_cast<const uint8_t*>(w[0]);
    p.w[1] = static_cast<const uint8_t*>(w[nmat == 2 ? 1 : 0]);
    p.msc = p.mbi = nullptr;
    p.mgshift = 0;
    p.row_bytes = weight_row_bytes(fmt, K);
    p.next_units = 0;
    p.next_groups = p.next_nmat = p.next_ctas = 1;
    if (next && next->units > 0) {
        p.next_tmap[0] = next->tmap[0];
        p.next_tmap[1] = next->tmap[next->nmat == 2 ? 1 : 0];
        p.next_units = next->units;
        p.next_groups = next->groups;
        p.next_nmat = next->nmat;
        p.next_ctas = next->units < sm_count ? next->units : sm_count;
    }
    p.x = x;
    p.y = y;
    p.fault = fault;
    p.N = N;
    p.K = K;
    p.tiles = (N + kTileRows - 1) / kTileRows;
    p.groups = K / kGroupK;
    p.units = p.tiles * p.groups * nmat;
    p.x_bf16 = x_bf16;
    p.y_bf16 = y_bf16;
    const int ctas = p.units < sm_count ? p.units : sm_count;
    // the 8-bit form needs every K-group of a CTA's unit range in its table
    const bool f8 = ntok == 1 && table_fits(nmat, p.units, p.groups, sm_count);
    auto kernel = fmt == kFmtQ4K ? (f8 ? (x_bf16 ? qmv_q4_k_tc_e4m3_kernel<2> : qmv_q4_k_tc_e4m3_kernel<3>)
                                       : qmv_q4_k_tc_kernel)
                  : f8 ? (x_bf16 ? (nmat == 2 ? qmv_q4_0_tc_e4m3_kernel<2, 2> : qmv_q4_0_tc_e4m3_kernel<1, 2>)
                                 : (nmat == 2 ? qmv_q4_0_tc_e4m3_kernel<2, 3> : qmv_q4_0_tc_e4m3_kernel<1, 3>))
                  : (nmat == 2 ? qmv_q4_0_tc_kernel<2, 1>
                               : (ntok == 2 ? qmv_q4_0_tc_kernel<1, 2> : qmv_q4_0_tc_kernel<1, 1>));
    return launch_qtc(kernel, p, ctas, stream);
}

// The mixed-bit forms take what the Q4_0 path takes (K % 256 == 0, tile and
// CTA limits) and an activation table that holds every K-group of a CTA's
// unit range.
bool qmv_mix_tc_supported(int64_t N, int64_t K, int sm_count) {
    if (!qmv_tc_supported(1, N, K, sm_count)) return false;
    const int tiles = (int)((N + kTileRows - 1) / kTileRows), groups = (int)(K / kGroupK);
    return table_fits(1, tiles * groups, groups, sm_count);
}

// bits = 4, 2 or 8; groups of 2^gshift weights (gshift >= 5).  tmaps: the
// codes ([N][K b / 64] 8-byte words, box (4 b, 128) or for int8 (16, 128), the
// 128- or 64-byte swizzle), and for groups of 32 the scales and, for int4,
// the biases ([N][K / 128] 8-byte words, box (2, 128)); qp, sc and bi the same
// arrays (sc and bi read directly for larger groups and for the read-back
// correction); bf16 x (two pieces) or fp32 x (three; int2 and int4 then read
// their scales directly, as the third pieces take the B2 region).
cudaError_t launch_qmv_mix_tc(int bits, const CUtensorMap* tmaps, const void* qp, const void* sc, const void* bi,
                              int gshift, const void* x, int x_bf16, void* y, int y_bf16, int N, int K,
                              int sm_count, unsigned int* fault, cudaStream_t stream) {
    if (bits != 2 && bits != 4 && bits != 8) return cudaErrorInvalidValue;
    if (gshift < 5 || (K >> gshift) << gshift != K) return cudaErrorInvalidValue;
    QtcParams p;
    p.tmap_w[0] = tmaps[0];
    p.tmap_w[1] = tmaps[gshift == 5 ? 1 : 0];
    p.tmap_bi = tmaps[gshift == 5 && bits == 4 ? 2 : 0];
    p.w[0] = p.w[1] = static_cast<const uint8_t*>(qp);
    p.msc = static_cast<const uint16_t*>(sc);
    p.mbi = static_cast<const uint16_t*>(bits == 4 ? bi : sc);
    p.mgshift = gshift;
    p.row_bytes = (int64_t)K * bits / 8;
    p.next_units = 0;
    p.next_groups = p.next_nmat = p.next_ctas = 1;
    p.x = x;
    p.y = y;
    p.fault = fault;
    p.N = N;
    p.K = K;
    p.tiles = (N + kTileRows - 1) / kTileRows;
    p.groups = K / kGroupK;
    p.units = p.tiles * p.groups;
    p.x_bf16 = x_bf16;
    p.y_bf16 = y_bf16;
    if (!table_fits(1, p.units, p.groups, sm_count)) return cudaErrorInvalidValue;
    auto kernel = x_bf16 ? (bits == 4 ? qmv_mix4_tc_e4m3_kernel<2>
                                      : (bits == 2 ? qmv_mix2_tc_e4m3_kernel<2> : qmv_mix8_tc_e4m3_kernel<2>))
                         : (bits == 4 ? qmv_mix4_tc_e4m3_kernel<3>
                                      : (bits == 2 ? qmv_mix2_tc_e4m3_kernel<3> : qmv_mix8_tc_e4m3_kernel<3>));
    return launch_qtc(kernel, p, p.units < sm_count ? p.units : sm_count, stream);
}

}  // namespace qbw
