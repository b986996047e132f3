// qmv_chain.cu -- a chain of Q4_0 matrix-vector products in one cooperative
// launch: step s computes y_s = W_s x_s (or the fused gate+up,
// gelu_tanh(Wg x_s) * (Wu x_s)), and x_s may be the output of an earlier step.
// One token's decode weight sweep (per layer: q|k|v, o, gate+up, down) is one
// such chain.
//
// Each step is the tensor-core kernel's 8-bit operand form (qmv_tc.cu,
// qmv_tc_common.cuh) over the step's own stream-K split of its units among
// the CTAs.  What the chain adds to a sequence of separate launches:
// * The copy warp streams every step's weights in one sequence.  Weights never
//   depend on activations, so it runs ahead across step boundaries and HBM
//   stays busy while the CTAs meet between steps.
// * After writing its share of step s's outputs, each CTA's dequantizing warps
//   pass a grid barrier: one thread adds 1 to a counter (release) and spins,
//   bounded, until all CTAs have (acquire).  They then rebuild the activation
//   table from x_{s+1}, reading through L2, since other CTAs just wrote it.
// * Split-tile shares live in the chain's own scratch; every finisher
//   consumes (zeroes) its contributors' words before the barrier, so each
//   step finds the scratch zero.
// The launch is cooperative: all CTAs are resident together, which the grid
// barrier requires.
#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "qbw_device.cuh"
#include "qbw_internal.h"
#include "qmv_tc_common.cuh"
#include "tc_common.cuh"

namespace qbw {
namespace {

using namespace qtc;

struct ChainParams {
    const ChainStepDesc* steps;
    unsigned int* fault;
    unsigned int* bar_count;          // [0] grid barrier counter, [1] abort flag; zero at launch
    unsigned long long* share;        // [ctas][2][128] split-tile shares
    int32_t nsteps;
};

constexpr int kDequantThreads = kProducerWarp * 32;     // warps 0 .. 11

__device__ __forceinline__ void dequant_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"(kDequantThreads) : "memory");
}

// The run's abort flag: set after any failed wait, so that every wait on
// another CTA (shares, grid barrier) returns at once instead of running out
// its own bound, and a broken run ends within about one bound.
__device__ __forceinline__ bool aborted(const unsigned int* flag) {
    return *static_cast<const volatile unsigned int*>(flag) != 0u;
}
__device__ __forceinline__ void set_abort(unsigned int* flag) { atomicExch(flag, 1u); }

// All CTAs have arrived `target` times in total.  Called by one thread per
// CTA after its step outputs are written; bounded.
__device__ __forceinline__ bool grid_barrier(unsigned int* count, unsigned int target, unsigned int* fault) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
        if (v >= target) return true;
        if (aborted(count + 1)) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            record_fault(fault, kFaultGridWait);
            return false;
        }
    }
}

// a split tile's share from another CTA (a word carrying this run's launch
// tag; a stale word from a run that faulted is never taken), unless the run
// has been aborted
__device__ __forceinline__ unsigned long long wait_share(const unsigned long long* src, uint32_t tag,
                                                         unsigned int* fault, unsigned int* abort_flag) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(src) : "memory");
    if ((uint32_t)(w >> 32) == tag) return w;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(src) : "memory");
        if ((uint32_t)(w >> 32) == tag) return w;
        if (aborted(abort_flag)) return w;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            record_fault(fault, kFaultShareWaitTimeout);
            set_abort(abort_flag);
            return w;
        }
    }
}

// A step descriptor's scalar fields (the 64 bytes after its two tensor maps),
// as the decode warps keep them in shared memory.
struct StepScalars {
    const void* x;
    void* y;
    const uint8_t* w[2];
    int32_t N, K, nmat, y_bf16;
    int32_t tiles, groups, units, reserved;
};
static_assert(sizeof(StepScalars) == 64 && offsetof(ChainStepDesc, x) == 2 * sizeof(CUtensorMap) &&
                  offsetof(ChainStepDesc, reserved) == offsetof(ChainStepDesc, x) + 60,
              "StepScalars mirrors the fields of ChainStepDesc after its tensor maps");

__device__ __forceinline__ void cp_async4_sh(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// the step's unit range of this CTA and its first and last tiles
struct StepRange {
    int G, nmat, GU, u0, u1, n, tile0, tile1;
    bool contrib0, fin1;
    template <typename Desc>
    __device__ __forceinline__ void init(const Desc& st, int cta, int ctas) {
        G = st.groups;
        nmat = st.nmat;
        GU = G * nmat;
        u0 = unit_begin(cta, st.units, ctas);
        u1 = unit_begin(cta + 1, st.units, ctas);
        n = u1 - u0;
        tile0 = u0 / GU;
        tile1 = n > 0 ? (u1 - 1) / GU : tile0;
        contrib0 = n > 0 && tile0 * GU < u0;
        fin1 = n > 0 && (tile1 + 1) * GU > u1 && tile1 * GU >= u0;
    }
};

__global__ void __launch_bounds__(kThreads, 1) qmv_chain_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ctas = (int)gridDim.x, cta = (int)blockIdx.x;
    const uint32_t tag = launch_tag();     // marks this run's split-tile shares
    __shared__ unsigned int qcount[4];
    if (threadIdx.x < 4) qcount[threadIdx.x] = 0u;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + kOffBar;
    float* part = reinterpret_cast<float*>(smem + kOffPart);      // [set][local tile][matrix][row]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
    bool ok = true;

    for (int i = threadIdx.x; i < (int)(kSets * kBBytes / 16); i += kThreads)
        sts128(sbase + kOffB + 16u * (uint32_t)i, make_uint4(0u, 0u, 0u, 0u));
    for (int i = threadIdx.x; i < kSets * kMaxLocalTiles * 2 * kTileRows; i += kThreads) part[i] = 0.f;
    for (int i = threadIdx.x; i < kProducerWarp * 32 * 3; i += kThreads)       // acc_q and fixups
        reinterpret_cast<uint32_t*>(smem + kOffQ)[i] = 0u;

    // this CTA's units over all steps (the ring and set sequence runs on across steps)
    int n_total = 0;
    for (int s = 0; s < p.nsteps; ++s) {
        const int U = p.steps[s].units;
        n_total += unit_begin(cta + 1, U, ctas) - unit_begin(cta, U, ctas);
    }

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
            // every step's weight rows, in order: I counts this CTA's units over all steps
            int I = 0;
            for (int s = 0; s < p.nsteps && ok; ++s) {
                const ChainStepDesc& st = p.steps[s];
                StepRange r;
                r.init(st, cta, ctas);
                prefetch_tmap(&st.tmap[0]);
                if (r.nmat == 2) prefetch_tmap(&st.tmap[1]);
                for (int i = 0; i < r.n; ++i, ++I) {
                    const int stg = I % kStages;
                    if (I >= kStages)
                        ok = mbar_wait_bounded(empty_bar(bar0, stg), (uint32_t)((I / kStages) - 1) & 1u, p.fault,
                                               kFaultBulkWaitTimeout);
                    if (!ok) {
                        set_abort(p.bar_count + 1);
                        break;
                    }
                    const int u = r.u0 + i, ug = u / r.nmat, mat = u - ug * r.nmat, t = ug / r.G, g = ug - t * r.G;
                    mbar_arrive_expect_tx(full_bar(bar0, stg), kRawStageBytes);
                    tma_load_2d(sbase + (uint32_t)stg * kRawStageBytes, &st.tmap[mat], g * kGroupWords,
                                t * kTileRows, full_bar(bar0, stg), policy_evict_first());
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
    // the first step's x belongs to the preceding grid's stream order
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp >= kMmaWarp0) {
        // ---------------- MMA issuer of set s: the set's units of every step
        const int set = warp - kMmaWarp0;
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(kTileRows, kN);
            const uint32_t a_tmem = tmem + (uint32_t)set * kACols;
            const uint64_t b0 = sw128_desc(sbase + kOffB + (uint32_t)set * kBBytes);
            uint32_t phase = 0;
            for (int I = set; I < n_total; I += kSets) {
                const uint32_t d_tmem = tmem + kDCol + 32u * (uint32_t)set + 16u * phase;
                ok = mbar_wait_bounded(afull_bar(bar0, set, 0), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) {
                    set_abort(p.bar_count + 1);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + (uint64_t)((k >> 2) * 128 + (k & 3) * 2),
                              idesc, k > 0 ? 1u : 0u);
                tc_commit(aempty_bar(bar0, set, 0));
                ok = mbar_wait_bounded(afull_bar(bar0, set, 1), phase, p.fault, kFaultMmaWaitTimeout);
                if (!ok) {
                    set_abort(p.bar_count + 1);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 8; k < 16; ++k)
                    tc_mma_f8(d_tmem, a_tmem + 8u * (uint32_t)k, b0 + (uint64_t)((k >> 2) * 128 + (k & 3) * 2),
                              idesc, 1u);
                tc_commit(aempty_bar(bar0, set, 1));
                phase ^= 1u;
            }
            tc_commit(done_bar(bar0));
        }
    } else if (warp < kProducerWarp) {
        // ---------------- dequantizing warp: set s, lane quarter q.  Every
        // warp executes every dequant_sync of every step, also after a failed
        // wait (it then only skips the work), so no barrier waits forever.
        const int set = warp >> 2, q = warp & 3;
        const uint32_t tmem = *tmem_slot;
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        const uint32_t a_taddr = tmem + lanes + (uint32_t)set * kACols;
        const uint32_t d_taddr = tmem + lanes + kDCol + 32u * (uint32_t)set;   // + 16 (k % 2)
        const uint32_t raw_row = (uint32_t)(32 * q + lane) * 144u;
        const uint32_t bbuf = sbase + kOffB + (uint32_t)set * kBBytes;
        // lanes 0..7 of warp q write B slots 8q .. 8q + 7 (blocks 2q, 2q + 1):
        // K-steps 2j (+x) and 2j + 1 (-x), rows 2j (piece 0) and 2j + 1 (piece 1)
        const int xl = 8 * q + lane;
        const bool bwriter = lane < 8;
        const int bj = xl >> 2, bhalf = xl >> 4;
        const uint32_t bo = (uint32_t)((bj & 1) * 64 + 8 * (xl & 3));
        const uint32_t f8_p0 = bbuf + b_byte(bj >> 1, 2 * bj, bo), f8_p1 = bbuf + b_byte(bj >> 1, 2 * bj + 1, bo);
        const uint32_t f8_n0 = bbuf + b_byte(bj >> 1, 2 * bj, bo + 32u);
        const uint32_t f8_n1 = bbuf + b_byte(bj >> 1, 2 * bj + 1, bo + 32u);
        const int row = 32 * q + lane;
        int I_base = 0;     // this CTA's units in the earlier steps
        int k = 0;          // the set's units so far, over all steps
        // Step s's scalar fields in slot s % 2 of a 128-byte cache in the second
        // B buffer (which the bf16 8-bit form leaves unused): threads 0..15 copy
        // step s + 1's while step s runs, and wait for them before the step's
        // last barrier, so no step starts on a read of device memory.
        const uint32_t dcache = sbase + kOffB2;
        auto fetch_scalars = [&](int s2) {
            if (threadIdx.x < 16 && s2 < p.nsteps)
                cp_async4_sh(dcache + 64u * (uint32_t)(s2 & 1) + 4u * threadIdx.x,
                             reinterpret_cast<const uint32_t*>(&p.steps[s2].x) + threadIdx.x);
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        fetch_scalars(0);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        dequant_sync();
        for (int s = 0; s < p.nsteps; ++s) {
            const StepScalars& st = *reinterpret_cast<const StepScalars*>(smem + kOffB2 + 64u * (uint32_t)(s & 1));
            fetch_scalars(s + 1);
            StepRange r;
            r.init(st, cta, ctas);
            const int G = r.G, nmat = r.nmat, u0 = r.u0, n = r.n, tile0 = r.tile0;
            const int xg0 = n > 0 ? (u0 / nmat) % G : 0;
            {
                const int cnt = n > 0 ? min(G, (r.u1 - 1) / nmat - u0 / nmat + 1) : 0;
                if (cnt > kXtGroups) record_fault(p.fault, kFaultPlan);
                build_x_table<true, 2>(sbase, st.x, xg0, G, min(cnt, kXtGroups), warp, lane, kProducerWarp);
            }
            dequant_sync();     // table written; part[] and qcount clear
            bool counted = !r.contrib0;
            // after the three sets' shares of the first tile are in part[][0][],
            // the last of a quarter's three warps publishes the quarter's rows
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
                    for (int m = 0; m < 2; ++m) {
                        if (m >= nmat) break;
                        const float v = part[part_at(0, 0, m, row)] + part[part_at(1, 0, m, row)] +
                                        part[part_at(2, 0, m, row)];
                        st_relaxed_u64(p.share + ((size_t)cta * 2 + m) * kTileRows + row,
                                       (unsigned long long)__float_as_uint(v) | ((unsigned long long)tag << 32));
                    }
                }
                counted = true;
            };
            // the row's sums of the tile being accumulated, one per matrix, and
            // the error-check terms of its flagged units
            float acc[2] = {0.f, 0.f};
            float* acc_q = reinterpret_cast<float*>(smem + kOffQ) + 2 * threadIdx.x;
            uint32_t* fixups = reinterpret_cast<uint32_t*>(smem + kOffFix) + threadIdx.x;
            int acc_tile = -1, pend_tile = -1, pend_mat = 0, pend_sl = 0;
            uint32_t pend_dd[4] = {0u, 0u, 0u, 0u};
            bool pend = false;
            // the exact sum of w r over this set's units of tile T, matrix m (r:
            // what the pieces miss), for a segment the check flags
            auto segment_correction = [&](int T, int m) -> float {
                const int64_t nrow = (int64_t)T * kTileRows + row;
                float corr = 0.f;
                if (nrow >= st.N) return corr;
                const int64_t rb = weight_row_bytes(kFmtQ4, st.K);
                for (int i = ((set - I_base) % kSets + kSets) % kSets; i < n; i += kSets) {
                    const int u = u0 + i, ug = u / nmat, mat = u - ug * nmat, t = ug / G, g = ug - t * G;
                    if (t > T) break;
                    if (t < T || mat != m) continue;
                    int sl = g - xg0;
                    if (sl < 0) sl += G;
                    if (sl >= kXtGroups) sl = 0;
                    if (!group_flagged(sbase, sl)) continue;     // no residuals
                    corr += unit_correction<kFmtQ4, 2, true>(st.w[m] + nrow * rb + (int64_t)g * 144, st.x, g, sbase, sl);
                }
                return corr;
            };
            // the set's partial rows of acc_tile -> part[]; a segment that fails
            // the error check (its units' terms, summed in acc_q) gets bit
            // 2 (acc_tile - tile0) + m in fixups, and its exact correction is
            // added after the step's unit loop
            auto flush = [&]() {
                if (acc_tile < 0) return;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const float q = acc_q[m];
                    if (q != 0.f) {
                        acc_q[m] = 0.f;
                        if (segment_needs_correction(q)) *fixups |= 1u << (2 * (acc_tile - tile0) + m);
                    }
                    part[part_at(set, acc_tile - tile0, m, row)] = acc[m];
                }
            };
            auto add_unit = [&](float r0) {
                if (pend_tile != acc_tile) {
                    flush();
                    acc[0] = 0.f;
                    acc[1] = 0.f;
                    acc_tile = pend_tile;
                    // a first-tile share that needs its correction is published
                    // after the unit loop instead
                    if (!counted && pend_tile > tile0 && !__any_sync(0xffffffffu, (*fixups & 3u) != 0u)) count_in();
                }
                if (pend_mat == 0) acc[0] += r0;
                else acc[1] += r0;
            };
            // D of the pending unit (buffer buf) -> its row sum
            auto read_back = [&](uint32_t buf) {
                uint32_t dv[16];
                tmem_ld16(d_taddr + 16u * buf, dv);
                tmem_wait_ld();
                float c[8];
                table_f8(sbase, kOffXc, pend_sl, c);
                const float r0 = unit_dot_e4m3(dv, pend_dd, c);
                add_unit(r0);
                if (__builtin_expect(__float_as_uint(c[0]) >> 31, 0)) {     // a flagged group
                    // the unit's error-check term into its segment's sum
                    float a[8];
                    table_f8(sbase, kOffXr, pend_sl, a);
                    acc_q[pend_mat] += unit_check_term<kFmtQ4>(dv, pend_dd, c, a);
                }
            };
            // this set's units of the step: I = I_base + i = set (mod 3)
            for (int i = ((set - I_base) % kSets + kSets) % kSets; i < n && ok; i += kSets, ++k) {
                const int I = I_base + i;
                const int u = u0 + i, ug = u / nmat, mat = u - ug * nmat, t = ug / G, g = ug - t * G;
                const int stg = I % kStages;
                // this unit's group in the table
                int cur_sl = g - xg0;
                if (cur_sl < 0) cur_sl += G;
                if (cur_sl >= kXtGroups) cur_sl = 0;       // never: the host checks the table size
                const bool got = mbar_wait_bounded(full_bar(bar0, stg), (uint32_t)(I / kStages) & 1u, p.fault,
                                                   kFaultBulkWaitTimeout);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    if (lane == 0) set_abort(p.bar_count + 1);
                    break;
                }
                const uint32_t src = sbase + (uint32_t)stg * kRawStageBytes + raw_row;
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
                if (lane == 0) mbar_arrive(empty_bar(bar0, stg));     // raw rows of the stage read
                uint32_t dd[4];
#pragma unroll
                for (int P = 0; P < 4; ++P) dd[P] = scale_pair(v, P);
                uint2 bp0 = make_uint2(0u, 0u), bp1 = bp0;
                if (bwriter) {
                    const uint4 tq = lds128(sbase + kOffXt + (uint32_t)(cur_sl * 32 + xl) * 16u);
                    bp0 = make_uint2(tq.x, tq.y);
                    bp1 = make_uint2(tq.z, tq.w);
                }
                const uint32_t prev = (uint32_t)(k - 1) & 1u;     // completion parity of the set's previous unit
                uint32_t c0[32], c1[32];
                // ---- half 0: K 0..127 (block pairs 0, 1; B atoms 0, 1 written by warps 0, 1)
                codes_pair_e4m3<0>(v, c0);
                if (k > 0) {
                    const bool free = mbar_wait_bounded(aempty_bar(bar0, set, 0), prev, p.fault,
                                                        kFaultMmaWaitTimeout);
                    if (!__all_sync(0xffffffffu, free)) {
                        ok = false;
                        if (lane == 0) set_abort(p.bar_count + 1);
                        break;
                    }
                    tc_fence_after();
                }
                if (bwriter && bhalf == 0) {
                    sts64(f8_p0, bp0);
                    sts64(f8_p1, bp1);
                    sts64(f8_n0, make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                    sts64(f8_n1, make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                    fence_proxy_async_smem();     // B visible to the tensor core
                }
                tmem_st32(a_taddr, c0);
                codes_pair_e4m3<1>(v, c1);
                tmem_wait_st();
                tmem_st32(a_taddr + 32u, c1);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(bar0, set, 0));
                // ---- half 1: K 128..255 (block pairs 2, 3; B atoms 2, 3 written by warps 2, 3)
                codes_pair_e4m3<2>(v, c0);
                if (k > 0) {
                    const bool free = mbar_wait_bounded(aempty_bar(bar0, set, 1), prev, p.fault,
                                                        kFaultMmaWaitTimeout);
                    if (!__all_sync(0xffffffffu, free)) {
                        ok = false;
                        if (lane == 0) set_abort(p.bar_count + 1);
                        break;
                    }
                    tc_fence_after();
                }
                if (bwriter && bhalf == 1) {
                    sts64(f8_p0, bp0);
                    sts64(f8_p1, bp1);
                    sts64(f8_n0, make_uint2(bp0.x ^ 0x80808080u, bp0.y ^ 0x80808080u));
                    sts64(f8_n1, make_uint2(bp1.x ^ 0x80808080u, bp1.y ^ 0x80808080u));
                    fence_proxy_async_smem();
                }
                tmem_st32(a_taddr + 64u, c0);
                codes_pair_e4m3<3>(v, c1);
                tmem_wait_st();
                tmem_st32(a_taddr + 96u, c1);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(bar0, set, 1));
                // the set's previous unit of this step (its D buffer is complete
                // since this unit's MMAs waited for its second half)
                if (pend) read_back(prev);
#pragma unroll
                for (int P = 0; P < 4; ++P) pend_dd[P] = dd[P];
                pend_sl = cur_sl;
                pend_tile = t;
                pend_mat = mat;
                pend = true;
            }
            if (ok && pend) {
                // the set's last unit of the step
                const uint32_t last = (uint32_t)(k - 1) & 1u;
                const bool fin = mbar_wait_bounded(aempty_bar(bar0, set, 1), last, p.fault, kFaultMmaWaitTimeout);
                if (__all_sync(0xffffffffu, fin)) {
                    tc_fence_after();
                    read_back(last);
                } else {
                    ok = false;
                    if (lane == 0) set_abort(p.bar_count + 1);
                }
            }
            flush();
            // the flagged segments' exact corrections (rare: activations whose
            // elements far below their block's largest carry the row's sum)
            uint32_t fx = *fixups;
            *fixups = 0u;
            while (fx != 0u) {
                const int b = __ffs(fx) - 1;
                fx &= fx - 1u;
                part[part_at(set, b >> 1, b & 1, row)] += segment_correction(tile0 + (b >> 1), b & 1);
            }
            if (!counted) count_in();
            dequant_sync();     // every set's partial rows are in part[]
            // ---- the step's tiles: whole ones -> y; the last one, when this CTA
            // covers its first unit but not its last, with the later CTAs' shares
            if (n > 0 && threadIdx.x < kTileRows) {
                const int rr = threadIdx.x;
                for (int t = tile0; t <= r.tile1; ++t) {
                    if (t == tile0 && r.contrib0) continue;                 // published already
                    const int lt = t - tile0;
                    float v[2];
#pragma unroll
                    for (int m = 0; m < 2; ++m)
                        v[m] = part[part_at(0, lt, m, rr)] + part[part_at(1, lt, m, rr)] + part[part_at(2, lt, m, rr)];
                    if (t == r.tile1 && r.fin1) {
                        // the later CTAs with units in the tile; a step with fewer
                        // units than CTAs leaves some CTAs without any (no share)
                        const int c_last = owner_of((t + 1) * r.GU - 1, st.units, ctas);
                        for (int c = cta + 1; c <= c_last; ++c) {
                            if (unit_begin(c + 1, st.units, ctas) == unit_begin(c, st.units, ctas)) continue;
#pragma unroll
                            for (int m = 0; m < 2; ++m) {
                                if (m >= nmat) break;
                                unsigned long long* src = p.share + ((size_t)c * 2 + m) * kTileRows + rr;
                                const unsigned long long w = wait_share(src, tag, p.fault, p.bar_count + 1);
                                v[m] += __uint_as_float((uint32_t)w);
                                st_relaxed_u64(src, 0ull);                 // consumed
                            }
                        }
                    }
                    const int64_t yrow = (int64_t)t * kTileRows + rr;
                    if (yrow < st.N) {
                        const float o = nmat == 2 ? gelu_tanh(v[0]) * v[1] : v[0];
                        if (st.y_bf16) store_out<__nv_bfloat16>(st.y, yrow, o);
                        else store_out<float>(st.y, yrow, o);
                    }
                }
            }
            dequant_sync();     // part[] read: clear it and the publish counters for the next step
            for (int i = threadIdx.x; i < kSets * kMaxLocalTiles * 2 * kTileRows; i += kDequantThreads) part[i] = 0.f;
            if (threadIdx.x < 4) qcount[threadIdx.x] = 0u;
            I_base += n;
            asm volatile("cp.async.wait_group 0;" ::: "memory");     // step s + 1's scalars landed
            if (s + 1 < p.nsteps) {
                // the step's outputs, written by every CTA, are the next steps' inputs
                __threadfence();
                dequant_sync();
                if (threadIdx.x == 0 && !grid_barrier(p.bar_count, (unsigned int)((s + 1) * ctas), p.fault)) {
                    ok = false;
                    set_abort(p.bar_count + 1);
                }
                dequant_sync();
            }
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
}

}  // namespace

// The step's unit split fits the kernel: at most kMaxLocalTiles tiles and
// kXtGroups activation-table groups per CTA.
bool qmv_chain_step_supported(int nmat, int64_t N, int64_t K, int ctas) {
    if (nmat < 1 || nmat > 2 || ctas < 1 || ctas > 1024) return false;
    if (K % kGroupK != 0 || K < kGroupK || N < 1) return false;
    const int64_t tiles = (N + kTileRows - 1) / kTileRows;
    const int64_t groups = K / kGroupK;
    const int64_t per_tile = groups * nmat;
    const int64_t units = tiles * per_tile;
    if (units > INT32_MAX) return false;
    const int64_t per = (units + ctas - 1) / ctas;
    return per / per_tile + 2 <= kMaxLocalTiles && std::min<int64_t>(groups, (per - 1) / nmat + 2) <= kXtGroups;
}

void qmv_chain_fill_step(ChainStepDesc* d, int nmat, int64_t N, int64_t K) {
    d->N = (int32_t)N;
    d->K = (int32_t)K;
    d->nmat = nmat;
    d->tiles = (int32_t)((N + kTileRows - 1) / kTileRows);
    d->groups = (int32_t)(K / kGroupK);
    d->units = d->tiles * d->groups * nmat;
    d->reserved = 0;
}

// CTAs of a chain launch on a device with sm_count SMs (0 if one CTA per SM
// does not fit)
int qmv_chain_ctas(int sm_count) {
    int per_sm = 0;
    if (cudaFuncSetAttribute(qmv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmv_chain_kernel, kThreads, kSmemBytes) !=
            cudaSuccess)
        return 0;
    return per_sm >= 1 ? sm_count : 0;
}

size_t qmv_chain_share_bytes(int ctas) { return (size_t)ctas * 2 * kTileRows * sizeof(unsigned long long); }

cudaError_t launch_qmv_chain(const ChainStepDesc* steps, int nsteps, int ctas, unsigned int* bar_count,
                             unsigned long long* share, unsigned int* fault, cudaStream_t stream) {
    ChainParams p;
    p.steps = steps;
    p.fault = fault;
    p.bar_count = bar_count;
    p.share = share;
    p.nsteps = nsteps;
    cudaError_t e = cudaMemsetAsync(bar_count, 0, 2 * sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qmv_chain_kernel, p);
}

}  // namespace qbw
