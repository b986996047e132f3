// api.cu -- the C ABI of libqbw (include/qbw.h): argument validation, the
// per-device capability cache, the launch planner of the streaming kernels and
// the entry points themselves.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "qbw.h"
#include "qbw_internal.h"

namespace qbw {

cudaError_t launch_stream_q4(int R, const StreamParams& p, int ctas, int warps, size_t smem, cudaStream_t s);
cudaError_t launch_stream_q8(int R, const StreamParams& p, int ctas, int warps, size_t smem, cudaStream_t s);
cudaError_t launch_stream_gateup(int R, const StreamParams& p, int ctas, int warps, size_t smem, cudaStream_t s);
cudaError_t prepare_stream_q4(int R, size_t smem);
cudaError_t prepare_stream_q8(int R, size_t smem);
cudaError_t prepare_stream_gateup(int R, size_t smem);
cudaError_t launch_qmm_generic(const uint8_t* w, const void* X, void* Y, int y_bf16, int64_t M, int64_t N,
                               int64_t K, int sm_count, cudaStream_t stream);
cudaError_t launch_qmm_tc(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x, void* y, int y_bf16, float* partials,
                          unsigned int* counters, unsigned long long* share, unsigned int* fault, int M, int N, int K,
                          int splits, int cluster, int streamk_ctas, cudaStream_t stream);
int qmm_tc_max_active_clusters(int nt, int cluster);
cudaError_t launch_selftest_wait(int which, uint64_t limit_ns, unsigned int* fault, cudaStream_t stream);
bool qmv_tc_supported(int nmat, int64_t N, int64_t K, int sm_count);
cudaError_t launch_qmv_tc(int fmt, int nmat, int ntok, const CUtensorMap* tmap_w, const void* const* w,
                          const void* x, int x_bf16, void* y, int y_bf16, int N, int K, int sm_count,
                          unsigned int* fault, cudaStream_t stream, const QtcNextLaunch* next = nullptr);
int qmm_tc_tile_rows();
bool qmv_mix_tc_supported(int64_t N, int64_t K, int sm_count);
cudaError_t launch_qmv_mix_tc(int bits, const CUtensorMap* tmaps, const void* qp, const void* sc, const void* bi,
                              int gshift, const void* x, int x_bf16, void* y, int y_bf16, int N, int K,
                              int sm_count, unsigned int* fault, cudaStream_t stream);
bool qmv_chain_step_supported(int nmat, int64_t N, int64_t K, int ctas);
void qmv_chain_fill_step(ChainStepDesc* d, int nmat, int64_t N, int64_t K);
int qmv_chain_ctas(int sm_count);
size_t qmv_chain_share_bytes(int ctas);
cudaError_t launch_qmv_chain(const ChainStepDesc* steps, int nsteps, int ctas, unsigned int* bar_count,
                             unsigned long long* share, unsigned int* fault, cudaStream_t stream);
int qmm_tc_group_k();

namespace {

// One fault word per device; kernels receive its address.
__device__ unsigned int g_fault_word = 0;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    size_t smem_optin = 0;
    unsigned int* fault = nullptr;
    // streaming-kernel instantiations whose shared-memory limit was raised
    bool stream_prepared[3][9] = {};
    // co-resident clusters of the small-M kernel, + 1 (0: not asked yet),
    // by MMA width (16, 32) and cluster size (0 .. 8)
    int qmm_clusters[2][9] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

qbw_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QBW_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        int major = 0, minor = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return QBW_ECUDA;
        di.supported = (major == 10 && minor == 3);
        di.sm_count = sms;
        di.smem_optin = (size_t)optin;
        if (di.supported) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_fault_word) != cudaSuccess) return QBW_ECUDA;
            di.fault = static_cast<unsigned int*>(addr);
        }
        di.ready = true;
    }
    if (!di.supported) return QBW_EDEVICE;
    *out = &di;
    return QBW_OK;
}

bool valid_dtype(qbw_dtype t) { return t == QBW_F32 || t == QBW_BF16; }
size_t dtype_size(qbw_dtype t) { return t == QBW_F32 ? 4 : 2; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

// ------------------------------------------------------------------ planner
struct StreamPlan {
    int R = 0, warps = 0, depth = 0, ctas = 0;
    size_t smem = 0;
    StreamParams p{};
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct StageLayout {
    size_t half, mat, stage;
};
StageLayout stage_layout(int fmt, int nmat, int R) {
    return {stage_half_bytes(fmt, R), stage_mat_bytes(fmt, R), stage_bytes_of(fmt, nmat, R)};
}

// cuTensorMapEncodeTiled, fetched once from the driver.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// View a weight matrix as [N][row_bytes / 8] 8-byte words; box = (box_words, R).
bool encode_weight_map(CUtensorMap* m, const void* w, int64_t N, int64_t row_bytes, int fmt, int R) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_words(fmt), (cuuint32_t)R};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Choose rows per group R, warps per CTA W and ring depth D for one streaming
// call.  Every SM runs one CTA owning ceil(groups / SMs) groups at most; its
// (group, chunk) items are dealt round-robin to the W warps.  The estimate of
// the makespan: the busiest warp's work (a full chunk costs R pair-rows per
// lane, the short final chunk ceil(R * tail / 32) without activation reuse),
// times W (the warps share the SM), divided by how well the SM is fed: enough
// warps to hide latency, enough bytes in flight, activation reuse across R.
bool plan_stream(int fmt, int nmat, int64_t N, int64_t K, const DeviceInfo& di, StreamPlan* out) {
    const int64_t npairs = K / 64;
    const int nfull = (int)(npairs / 32);
    const int tail = (int)(npairs % 32);
    const int nitems = nfull + (tail ? 1 : 0);
    const size_t xs_bytes = (size_t)npairs * 68 * 4;   // 64 activations per pair, padded to 68
    const size_t fixed = align_up(xs_bytes, 128);
    const int Rs_1[] = {8, 4, 2, 1};
    const int Rs_2[] = {4, 2, 1};
    const int* Rs = (nmat == 2) ? Rs_2 : Rs_1;
    const int nR = (nmat == 2) ? 3 : 4;
    double best = 0.0;
    bool found = false;
    for (int ir = 0; ir < nR; ++ir) {
        const int R = Rs[ir];
        const size_t stage = stage_layout(fmt, nmat, R).stage;
        const int64_t groups = (N + R - 1) / R;
        const int64_t gmax = (groups + di.sm_count - 1) / di.sm_count;
        const int64_t items = gmax * nitems;
        const size_t part_bytes = align_up((size_t)items * nmat * R * 4, 128);
        const double full_cost = (double)R;
        const double tail_cost = tail ? 1.15 * (double)((R * tail + 31) / 32) : 0.0;
        for (int W = 16; W >= 4; --W) {
            double warp_cost[16] = {};
            for (int64_t it = 0; it < items; ++it)
                warp_cost[it % W] += ((it % nitems) < nfull) ? full_cost : tail_cost;
            double makespan = 0.0;
            for (int w = 0; w < W; ++w) makespan = std::max(makespan, warp_cost[w]);
            for (int D = 4; D >= 2; --D) {
                const size_t smem = fixed + (size_t)W * D * stage + (size_t)W * D * 8 + part_bytes + 128;
                if (smem > di.smem_optin) continue;
                const double sat = std::min(1.0, W / 12.0);
                const double lat = std::sqrt(std::min(1.0, (double)W * (D - 1) * (double)stage / 65536.0));
                const double reuse = 1.0 / (1.0 + 0.12 / R);
                const double t = makespan * W / (sat * lat * reuse);
                if (!found || t < best - 1e-9) {
                    found = true;
                    best = t;
                    out->R = R;
                    out->warps = W;
                    out->depth = D;
                    out->smem = smem;
                }
            }
        }
    }
    if (!found) return false;
    out->ctas = di.sm_count;
    StreamParams& p = out->p;
    const StageLayout L = stage_layout(fmt, nmat, out->R);
    const size_t stage = L.stage;
    p.row_bytes = (K / 32) * block_bytes(fmt);
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.npairs = (int32_t)npairs;
    p.ngroups = (int32_t)((N + out->R - 1) / out->R);
    p.nfull = nfull;
    p.tail_pairs = tail;
    p.depth = out->depth;
    p.ring_off = (uint32_t)fixed;
    p.stage_bytes = (uint32_t)stage;
    p.mat_bytes = (uint32_t)L.mat;
    p.half_bytes = (uint32_t)L.half;
    p.bar_off = (uint32_t)(fixed + (size_t)out->warps * out->depth * stage);
    p.part_off = (uint32_t)(p.bar_off + (size_t)out->warps * out->depth * 8);
    {
        const int64_t groups = (N + out->R - 1) / out->R;
        const int64_t gmax = (groups + di.sm_count - 1) / di.sm_count;
        p.slot_off = (uint32_t)(p.part_off + align_up((size_t)gmax * nitems * nmat * out->R * 4, 128));
    }
    p.fault = di.fault;
    return true;
}

// X [M][K] bf16 row-major as a 2-D tensor; box (64, nt) with the 128-byte
// swizzle of the tensor-core B operand.
// Q4_0 rows as 8-byte words in 128-row tiles of one 256-element K-group
// (144 bytes per row): the raw-weight box of the tensor-core kernels.  No L2
// promotion: a row's 144-byte segment then fetches only its own sectors
// (with 256-byte promotion the fused gate+up read 137.6 MB per 130.1 MB of
// weights, without it 134.9 MB, and ran 1 % faster).
bool encode_q4_tile_map(CUtensorMap* m, const void* w, int64_t N, int64_t K) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)((K / 32) * 18 / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)((K / 32) * 18)};
    cuuint32_t box[2] = {(cuuint32_t)(144 / 8), (cuuint32_t)qmm_tc_tile_rows()};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(w), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The int4-affine (bits = 4), int2-symmetric (bits = 2) or int8 (bits = 8)
// mixed-bit matrices with groups of 32, for the tensor-core kernel: m[0] the
// codes as [N][K b / 64] 8-byte words, box (4 b, 128) (one 256-element K-group
// of a 128-row tile, 32 b bytes per row; int8: half of it, 128 bytes, per
// copy) with the 128-byte (int4, int8) or 64-byte (int2) swizzle; m[1] and,
// for int4, m[2] the fp16 scales and biases as [N][K / 128] 8-byte words, box
// (2, 128) (the group's 8 of each per row; larger groups' scales and biases
// are read by the kernel's threads, without a map).  Needs K % 256 == 0 and
// 16-byte aligned arrays.
bool encode_mix_maps(CUtensorMap* m, int bits, const void* qp, const void* sc, const void* bi, int64_t N,
                     int64_t K, int64_t group) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t rows = (cuuint32_t)qmm_tc_tile_rows();
    cuuint32_t estr[2] = {1, 1};
    {
        cuuint64_t dims[2] = {(cuuint64_t)(K * bits / 64), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K * bits / 8)};
        cuuint32_t box[2] = {(cuuint32_t)(bits == 8 ? 16 : 4 * bits), rows};      // 256 weights of b bits (int8: 128)
        if (enc(&m[0], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(qp), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, bits == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    const void* sb[2] = {sc, bi};
    for (int i = 0; i < (group != 32 ? 0 : bits == 4 ? 2 : 1); ++i) {
        cuuint64_t dims[2] = {(cuuint64_t)(K / 128), (cuuint64_t)N};
        cuuint64_t strides[1] = {(cuuint64_t)(K / 16)};
        cuuint32_t box[2] = {2, rows};
        if (enc(&m[1 + i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(sb[i]), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool encode_x_map(CUtensorMap* m, const void* X, int64_t M, int64_t K, int nt) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)(K * 2)};
    cuuint32_t box[2] = {64, (cuuint32_t)nt};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split-K plan of the tensor-core small-M kernel: 128-row tiles, each split
// over `splits` CTAs (at most one CTA per SM in all), K-groups of 256.
//
// Workspace layout, the same for every shape so that one workspace can serve
// calls of different shapes: the tile arrival counters first, in a fixed
// region of kQmmCounterBytes, then the partial sums (or, for a stream-K plan,
// the CTAs' tagged shares).  Each call leaves the whole workspace zero again:
// counters reset, partial sums cleared, shares' tags cleared by the finishing
// CTA.
constexpr size_t kQmmCounterBytes = 4096;
//
// With 2 .. 8 splits per tile, and room on the device for all tiles' clusters
// at once, the splits of a tile run as one cluster and add their partial sums
// in distributed shared memory: no workspace.
constexpr int kQmmMaxCluster = 8;
struct QmmPlan {
    bool tc = false, cluster = false;
    bool exact = false;    // one or two token rows on the exact-code M = 1 kernel (qmv_tc.cu)
    int tiles = 0, splits = 1;
    int streamk_ctas = 0;  // > 0: stream-K over this many CTAs (one per SM), shares at share_off
    size_t partial_off = 0, share_off = 0, workspace = 0;
};

int qmm_clusters_fit(DeviceInfo& di, int nt, int cluster) {
    std::lock_guard<std::mutex> lk(g_mu);
    int& c = di.qmm_clusters[nt > 16 ? 1 : 0][cluster];
    if (c == 0) c = qmm_tc_max_active_clusters(nt, cluster) + 1;
    return c - 1;
}

QmmPlan plan_qmm(int64_t M, int64_t N, int64_t K, DeviceInfo& di) {
    QmmPlan q;
    if (M < 1 || M > 32 || K % 256 != 0 || N < 1) return q;
    // One or two tokens: the exact-code kernel carries them in its per-block
    // B columns at the cost of one (same size threshold as qmv_q4_0).
    if (M <= 2 && (double)N * (double)(K / 32) * 18.0 >= 15e6 && qmv_tc_supported(1, N, K, di.sm_count)) {
        q.tc = true;
        q.exact = true;
        return q;
    }
    q.tc = true;
    q.tiles = (int)((N + qmm_tc_tile_rows() - 1) / qmm_tc_tile_rows());
    const int groups = (int)(K / qmm_tc_group_k());
    int splits = di.sm_count / q.tiles;
    if (splits < 1) splits = 1;
    if (splits > groups) splits = groups;
    // Stream-K (M <= 16, so that two segments' accumulators fit TMEM): one CTA
    // per SM over equal ranges of the (tile, K-group) units.  It pays for its
    // tagged-share finish (measured at 2 to 4 us) only on long ranges (at least
    // 16 groups a CTA), where whole-tile splits add partial sums anyway (two
    // or more splits) and the busiest CTA then runs at least two and an eighth
    // fewer groups.  With fewer tiles than SMs no range is longer than a tile.
    const int64_t units = (int64_t)q.tiles * groups;
    const int ctas = di.sm_count;
    const int64_t busiest_split = (groups + splits - 1) / splits, busiest_streamk = (units + ctas - 1) / ctas;
    if (M <= 16 && splits >= 2 && q.tiles < ctas && units >= 16 * (int64_t)ctas &&
        busiest_split - busiest_streamk >= 2 && 8 * busiest_streamk <= 7 * busiest_split) {
        q.streamk_ctas = ctas;
        q.share_off = kQmmCounterBytes;
        // shares [ctas][M rounded up to 4][128 rows] of 64-bit tagged words
        const size_t mp = (size_t)((M + 3) / 4 * 4);
        q.workspace = kQmmCounterBytes + align_up((size_t)ctas * mp * (size_t)qmm_tc_tile_rows() * 8, 256);
        return q;
    }
    if (splits >= 2 && splits <= kQmmMaxCluster &&
        qmm_clusters_fit(di, (int)((M + 15) / 16 * 16), splits) >= q.tiles) {
        q.splits = splits;
        q.cluster = true;
        return q;
    }
    if ((size_t)q.tiles * 4 > kQmmCounterBytes) splits = 1;
    q.splits = splits;
    if (splits > 1) {
        q.partial_off = kQmmCounterBytes;
        // partial tiles [split][tile][128 rows][M rounded up to 4] fp32
        const size_t mp = (size_t)((M + 3) / 4 * 4);
        q.workspace = kQmmCounterBytes +
                      align_up((size_t)splits * (size_t)q.tiles * (size_t)qmm_tc_tile_rows() * mp * 4, 256);
    }
    return q;
}

int r_index(int R) { return R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3; }

// Plans are a pure function of (format, matrices, N, K) on a device, and the
// search above is not free on the host, so the last few are kept per device.
constexpr int kPlanCache = 16;
struct PlanEntry {
    bool valid = false, ok = false;
    int fmt = 0, nmat = 0;
    int64_t N = 0, K = 0;
    StreamPlan plan;
};
PlanEntry g_plans[kMaxDevices][kPlanCache];
int g_plan_next[kMaxDevices] = {};

bool plan_stream_cached(int fmt, int nmat, int64_t N, int64_t K, const DeviceInfo& di, StreamPlan* out) {
    const int dev = (int)(&di - g_dev);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (const PlanEntry& e : g_plans[dev])
            if (e.valid && e.fmt == fmt && e.nmat == nmat && e.N == N && e.K == K) {
                if (e.ok) *out = e.plan;
                return e.ok;
            }
    }
    StreamPlan plan;
    const bool ok = plan_stream(fmt, nmat, N, K, di, &plan);
    std::lock_guard<std::mutex> lk(g_mu);
    PlanEntry& e = g_plans[dev][g_plan_next[dev]++ % kPlanCache];
    e.valid = true;
    e.ok = ok;
    e.fmt = fmt;
    e.nmat = nmat;
    e.N = N;
    e.K = K;
    e.plan = plan;
    if (ok) *out = plan;
    return ok;
}

qbw_status launch_streaming(int fmt, int nmat, DeviceInfo& di, const StreamPlan& plan, cudaStream_t s) {
    const int which = (nmat == 2) ? 2 : (fmt == kFmtQ4 ? 0 : 1);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        bool& prepared = di.stream_prepared[which][r_index(plan.R)];
        if (!prepared) {
            cudaError_t e = (which == 0)   ? prepare_stream_q4(plan.R, di.smem_optin)
                            : (which == 1) ? prepare_stream_q8(plan.R, di.smem_optin)
                                           : prepare_stream_gateup(plan.R, di.smem_optin);
            if (e != cudaSuccess) return QBW_ECUDA;
            prepared = true;
        }
    }
    cudaError_t e = (which == 0)   ? launch_stream_q4(plan.R, plan.p, plan.ctas, plan.warps, plan.smem, s)
                    : (which == 1) ? launch_stream_q8(plan.R, plan.p, plan.ctas, plan.warps, plan.smem, s)
                                   : launch_stream_gateup(plan.R, plan.p, plan.ctas, plan.warps, plan.smem, s);
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

// Shared body of the three M = 1 entry points.
qbw_status qmv_common(int fmt, int nmat, const void* w0, const void* w1, const void* x, qbw_dtype xt, void* y,
                      qbw_dtype yt, int64_t M, int64_t N, int64_t K, void* stream) {
    if (!w0 || !x || !y || (nmat == 2 && !w1)) return QBW_EINVAL;
    if (!valid_dtype(xt) || !valid_dtype(yt)) return QBW_EDTYPE;
    if (M != 1) return QBW_ESHAPE;
    if (N < 1 || N > INT32_MAX || K < 32 || K % 32 != 0 || K > (int64_t(1) << 24)) return QBW_ESHAPE;
    if (fmt == kFmtQ4K && K % 256 != 0) return QBW_ESHAPE;
    if ((uintptr_t)x % dtype_size(xt) || (uintptr_t)y % dtype_size(yt)) return QBW_EALIGN;
    const size_t wbytes = (size_t)N * (size_t)weight_row_bytes(fmt, K);
    const size_t ybytes = (size_t)N * dtype_size(yt);
    if (overlaps(y, ybytes, x, (size_t)K * dtype_size(xt)) || overlaps(y, ybytes, w0, wbytes) ||
        (nmat == 2 && overlaps(y, ybytes, w1, wbytes)))
        return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool aligned = ((uintptr_t)w0 % 16 == 0) && (nmat == 1 || (uintptr_t)w1 % 16 == 0);
    // Q4_0 goes to the tensor cores from about 15 MB of weights (one matrix)
    // or 32 MB (gate + up); below that the streaming kernel's shorter start-up
    // wins (GB300, CUDA-graph replay: 5376 x 5376 8.3 vs 8.7 us, 4096 x 4096
    // 6.7 vs 6.1 us; gate+up 21504 x 5376 30.8 vs 34.4 us, 8192 x 2048 9.9 vs 8.3 us).
    // Q4_K has no streaming kernel: it takes the tensor cores whenever the
    // alignment allows, else the exact CUDA-core kernel.
    const bool tc_size = fmt == kFmtQ4K || (double)wbytes * nmat >= (nmat == 2 ? 32e6 : 15e6);
    if ((fmt == kFmtQ4 || fmt == kFmtQ4K) && tc_size && K % 256 == 0 && aligned && (uintptr_t)x % 16 == 0 &&
        qmv_tc_supported(nmat, N, K, di->sm_count)) {
        CUtensorMap tw[2];
        if (encode_q4_tile_map(&tw[0], w0, N, K) && (nmat == 1 || encode_q4_tile_map(&tw[1], w1, N, K))) {
            const void* wp[2] = {w0, nmat == 2 ? w1 : w0};
            cudaError_t e = launch_qmv_tc(fmt, nmat, 1, tw, wp, x, xt == QBW_BF16, y, yt == QBW_BF16, (int)N,
                                          (int)K, di->sm_count, di->fault, s);
            return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
        }
    }
    if (fmt != kFmtQ4K && K % 256 == 0 && aligned) {
        StreamPlan plan;
        if (plan_stream_cached(fmt, nmat, N, K, *di, &plan) &&
            encode_weight_map(&plan.p.tmap[0], w0, N, plan.p.row_bytes, fmt, plan.R) &&
            (nmat == 1 || encode_weight_map(&plan.p.tmap[1], w1, N, plan.p.row_bytes, fmt, plan.R))) {
            plan.p.w0 = static_cast<const uint8_t*>(w0);
            plan.p.w1 = static_cast<const uint8_t*>(nmat == 2 ? w1 : w0);
            plan.p.x = x;
            plan.p.y = y;
            plan.p.x_bf16 = (xt == QBW_BF16);
            plan.p.x_vec = ((uintptr_t)x % (xt == QBW_BF16 ? 8 : 16)) == 0;
            plan.p.y_bf16 = (yt == QBW_BF16);
            return launch_streaming(fmt, nmat, *di, plan, s);
        }
    }
    cudaError_t e = launch_qmv_generic(fmt, nmat, static_cast<const uint8_t*>(w0), static_cast<const uint8_t*>(w1),
                                       x, xt == QBW_BF16, y, yt == QBW_BF16, N, K, di->sm_count, s);
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

}  // namespace
}  // namespace qbw

// A built chain: its step descriptors, grid-barrier counter and split-tile
// scratch in device memory, on the device that was current at creation.
struct qbw_chain_s {
    int device = -1;
    int nsteps = 0;
    int ctas = 0;
    int sm_count = 0;
    std::vector<qbw::ChainStepDesc> host;   // the step descriptors, for runs as separate launches
    qbw::ChainStepDesc* steps = nullptr;
    unsigned int* bar = nullptr;          // [0] grid barrier counter, [1] abort flag
    unsigned long long* share = nullptr;
    unsigned int* fault = nullptr;
};

using namespace qbw;

extern "C" {

const char* qbw_status_str(qbw_status s) {
    switch (s) {
        case QBW_OK: return "QBW_OK";
        case QBW_EINVAL: return "QBW_EINVAL: null pointer, overlapping buffers or invalid argument";
        case QBW_ESHAPE: return "QBW_ESHAPE: M, N or K out of range (K must be a positive multiple of 32)";
        case QBW_EDTYPE: return "QBW_EDTYPE: unsupported activation or output dtype";
        case QBW_EALIGN: return "QBW_EALIGN: activation or output pointer not aligned to its dtype";
        case QBW_ECUDA: return "QBW_ECUDA: a CUDA call or kernel launch failed";
        case QBW_EWORKSPACE: return "QBW_EWORKSPACE: workspace missing, too small or misaligned";
        case QBW_EDEVICE: return "QBW_EDEVICE: current device is not compute capability 10.3";
    }
    return "QBW_?: unknown status";
}

uint32_t qbw_version(void) { return (1u << 16) | 0u; }

qbw_status qmv_q8_0(const void* w, const void* x, qbw_dtype xt, void* y, qbw_dtype yt, int64_t M, int64_t N,
                    int64_t K, void* stream) {
    return qmv_common(kFmtQ8, 1, w, nullptr, x, xt, y, yt, M, N, K, stream);
}

qbw_status qmv_q4_0(const void* w, const void* x, qbw_dtype xt, void* y, qbw_dtype yt, int64_t M, int64_t N,
                    int64_t K, void* stream) {
    return qmv_common(kFmtQ4, 1, w, nullptr, x, xt, y, yt, M, N, K, stream);
}

qbw_status qmv_q4_k(const void* w, const void* x, qbw_dtype xt, void* y, qbw_dtype yt, int64_t M, int64_t N,
                    int64_t K, void* stream) {
    return qmv_common(kFmtQ4K, 1, w, nullptr, x, xt, y, yt, M, N, K, stream);
}

qbw_status qmv_gateup_q4_0(const void* w_gate, const void* w_up, const void* x, qbw_dtype xt, void* out,
                           qbw_dtype ot, int64_t M, int64_t N, int64_t K, void* stream) {
    return qmv_common(kFmtQ4, 2, w_gate, w_up, x, xt, out, ot, M, N, K, stream);
}

size_t qmm_q4_0_smallM_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    DeviceInfo* di = nullptr;
    if (device_info(&di) != QBW_OK) return 0;
    return plan_qmm(M, N, K, *di).workspace;
}

qbw_status qmm_q4_0_smallM(const void* w, const void* X, qbw_dtype xt, void* Y, qbw_dtype yt, int64_t M,
                           int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    if (!w || !X || !Y) return QBW_EINVAL;
    if (xt != QBW_BF16 || !valid_dtype(yt)) return QBW_EDTYPE;
    if (M < 1 || M > 32 || N < 1 || N > INT32_MAX || K < 32 || K % 32 != 0 || K > (int64_t(1) << 24))
        return QBW_ESHAPE;
    if ((uintptr_t)X % 2 || (uintptr_t)Y % dtype_size(yt)) return QBW_EALIGN;
    const size_t ybytes = (size_t)M * N * dtype_size(yt);
    if (overlaps(Y, ybytes, X, (size_t)M * K * 2) || overlaps(Y, ybytes, w, (size_t)N * (K / 32) * 18))
        return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const QmmPlan q = plan_qmm(M, N, K, *di);
    if (q.exact && (uintptr_t)w % 16 == 0 && (uintptr_t)X % 16 == 0) {
        CUtensorMap tw[2];
        if (encode_q4_tile_map(&tw[0], w, N, K)) {
            const void* wp[2] = {w, w};
            cudaError_t e = launch_qmv_tc(kFmtQ4, 1, (int)M, tw, wp, X, 1, Y, yt == QBW_BF16, (int)N, (int)K,
                                          di->sm_count, di->fault, s);
            return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
        }
    }
    if (q.tc && !q.exact && (uintptr_t)w % 16 == 0 && (uintptr_t)X % 16 == 0) {
        if (q.workspace) {
            if (!workspace || workspace_bytes < q.workspace || (uintptr_t)workspace % 256) return QBW_EWORKSPACE;
            if (overlaps(workspace, q.workspace, Y, ybytes) || overlaps(workspace, q.workspace, X, (size_t)M * K * 2) ||
                overlaps(workspace, q.workspace, w, (size_t)N * (K / 32) * 18))
                return QBW_EINVAL;
        }
        CUtensorMap tw, tx;
        const int nt = (int)((M + 15) / 16 * 16);
        if (encode_q4_tile_map(&tw, w, N, K) && encode_x_map(&tx, X, M, K, nt)) {
            uint8_t* ws = static_cast<uint8_t*>(workspace);
            const bool sk = q.streamk_ctas > 0;
            cudaError_t e = launch_qmm_tc(
                tw, tx, Y, yt == QBW_BF16, q.workspace && !sk ? reinterpret_cast<float*>(ws + q.partial_off) : nullptr,
                q.workspace && !sk ? reinterpret_cast<unsigned int*>(ws) : nullptr,
                sk ? reinterpret_cast<unsigned long long*>(ws + q.share_off) : nullptr, di->fault, (int)M, (int)N,
                (int)K, q.splits, q.cluster ? 1 : 0, q.streamk_ctas, s);
            return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
        }
    }
    cudaError_t e = launch_qmm_generic(static_cast<const uint8_t*>(w), X, Y, yt == QBW_BF16, M, N, K, di->sm_count, s);
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

static qbw_status dequant_common(int fmt, const void* w, float* out, int64_t N, int64_t K, void* stream) {
    if (!w || !out) return QBW_EINVAL;
    if (N < 1 || K < 32 || K % 32 != 0 || K > (int64_t(1) << 24) || N > INT32_MAX) return QBW_ESHAPE;
    if (fmt == kFmtQ4K && K % 256 != 0) return QBW_ESHAPE;
    if ((uintptr_t)out % 4) return QBW_EALIGN;
    if (overlaps(out, (size_t)N * K * 4, w, (size_t)N * (size_t)weight_row_bytes(fmt, K))) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaError_t e = launch_dequant(fmt, static_cast<const uint8_t*>(w), out, N, K, di->sm_count,
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qdequant_q8_0(const void* w, float* out, int64_t N, int64_t K, void* stream) {
    return dequant_common(kFmtQ8, w, out, N, K, stream);
}

// Shared argument checks of the mixed-bit entry points: kind (2, 4, 8 bits),
// group G (a multiple of 16 dividing K), K (rows of whole 16-byte word groups,
// at most what the staged activations allow), pointers and alignment.
static qbw_status mixbit_args(qbw_mixbit kind, const void* qp, const void* sc, const void* bi, int64_t group,
                              int64_t N, int64_t K, size_t* wbytes) {
    const int bits = (int)kind;
    if (bits != 2 && bits != 4 && bits != 8) return QBW_EINVAL;
    if (!qp || !sc || (bits == 4 && !bi)) return QBW_EINVAL;
    if (N < 1 || N > INT32_MAX || K < 16 || K > (int64_t(1) << 24)) return QBW_ESHAPE;
    if (group < 16 || group % 16 != 0 || K % group != 0 || (K * bits) % 128 != 0) return QBW_ESHAPE;
    if ((uintptr_t)qp % 16 || (uintptr_t)sc % 4 || (bits == 4 && (uintptr_t)bi % 4)) return QBW_EALIGN;
    *wbytes = (size_t)N * (size_t)K * bits / 8;
    return QBW_OK;
}

// Bytes of codes from which the mixed-bit product takes the tensor cores:
// below them the CUDA-core kernel's shorter start-up wins, and more so for
// short rows (GB300, CUDA-graph replay, groups of 32, bf16 x, tensor cores vs
// CUDA cores; int4: 2048 x 5376 6.7 vs 7.7 us, 4096 x 4096 6.1 vs 6.0, 4096 x
// 2048 5.5 vs 3.5, 16384 x 2048 7.2 vs 8.5, 21504 x 5376 14.5 vs 27.3; int2:
// 2048 x 5376 6.7 vs 4.7, 3077 x 5376 6.7 vs 6.8, 4096 x 4096 6.0 vs 6.2,
// 4096 x 2048 5.4 vs 3.3, 16384 x 2048 7.1 vs 8.1, 21504 x 5376 13.5 vs 24.9;
// int8: 2048 x 5376 8.2 vs 8.3, 3077 x 5376 8.6 vs 8.7, 5376 x 5376 9.9 vs
// 12.8, 4096 x 4096 7.9 vs 6.6, 16384 x 2048 9.7 vs 9.0, 21504 x 5376 23.6 vs
// 29.9).
constexpr double mix_tc_min_bytes(int bits, int64_t K) {
    return bits == 8 ? (K > 4096 ? 16e6 : 64e6) : bits == 4 ? (K > 4096 ? 5e6 : 10e6) : (K > 4096 ? 4e6 : 5e6);
}

// Which kernel a mixed-bit product takes (shared by qmv_mixbit and
// qmv_mixbit_route).  Before the device is looked up: whether the call has the
// tensor-core form's shape (groups of 32 or a larger power of two, K % 256,
// size, scale alignment) and whether the CUDA-core kernel can stage its rows; after it,
// whether the device's plan takes the call and its tensor maps encode.
struct MixRoute {
    bool tc_form, cuda_fits;
};
static MixRoute mix_route(int bits, const void* sc, const void* bi, int64_t group, qbw_dtype xt, size_t wbytes,
                          int64_t K) {
    MixRoute r;
    r.tc_form = group >= 32 && (group & (group - 1)) == 0 && K % 256 == 0 &&
                (double)wbytes >= mix_tc_min_bytes(bits, K) &&
                (uintptr_t)sc % 16 == 0 && (bits != 4 || (uintptr_t)bi % 16 == 0);
    r.cuda_fits = qmv_mixbit_smem_bytes(bits, K, group) <= kMixMaxSmem;
    return r;
}
static bool mix_tc_maps(const MixRoute& r, int bits, const void* qp, const void* sc, const void* bi,
                        int64_t group, int64_t N, int64_t K, const DeviceInfo& di, CUtensorMap* maps) {
    return r.tc_form && qmv_mix_tc_supported(N, K, di.sm_count) &&
           encode_mix_maps(maps, bits, qp, sc, bi, N, K, group);
}

qbw_status qmv_mixbit(qbw_mixbit kind, const void* qp, const void* sc, const void* bi, int64_t group, const void* x,
                      qbw_dtype xt, void* y, qbw_dtype yt, int64_t M, int64_t N, int64_t K, void* stream) {
    size_t wbytes = 0;
    qbw_status st = mixbit_args(kind, qp, sc, bi, group, N, K, &wbytes);
    if (st != QBW_OK) return st;
    if (!x || !y) return QBW_EINVAL;
    if (!valid_dtype(xt) || !valid_dtype(yt)) return QBW_EDTYPE;
    if (M != 1) return QBW_ESHAPE;
    if ((uintptr_t)x % 16 || (uintptr_t)y % dtype_size(yt)) return QBW_EALIGN;
    const size_t ybytes = (size_t)N * dtype_size(yt), sbytes = (size_t)N * (size_t)(K / group) * 2;
    if (overlaps(y, ybytes, x, (size_t)K * dtype_size(xt)) || overlaps(y, ybytes, qp, wbytes) ||
        overlaps(y, ybytes, sc, sbytes) || (kind == QBW_MIXBIT_INT4_AFFINE && overlaps(y, ybytes, bi, sbytes)))
        return QBW_EINVAL;
    // groups of 32 (or a larger power of two): the tensor-core 8-bit form
    // (bf16 or fp32 x) from mix_tc_min_bytes of codes (where the device's plan
    // allows it); otherwise
    // the CUDA-core kernel, which stages x in shared memory, so its rows are
    // bounded
    const int bits = (int)kind;
    const MixRoute r = mix_route(bits, sc, bi, group, xt, wbytes, K);
    if (!r.tc_form && !r.cuda_fits) return QBW_ESHAPE;
    DeviceInfo* di = nullptr;
    st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CUtensorMap maps[3];
    if (mix_tc_maps(r, bits, qp, sc, bi, group, N, K, *di, maps)) {
        int gshift = 5;
        while ((int64_t(1) << gshift) < group) ++gshift;
        cudaError_t e = launch_qmv_mix_tc(bits, maps, qp, sc, bi, gshift, x, xt == QBW_BF16, y, yt == QBW_BF16,
                                          (int)N, (int)K, di->sm_count, di->fault, s);
        return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
    }
    if (!r.cuda_fits) return QBW_ESHAPE;
    cudaError_t e = launch_qmv_mixbit((int)kind, qp, sc, bi, (int)group, x, xt == QBW_BF16, y, yt == QBW_BF16, (int)N,
                                      (int)K, di->sm_count, s);
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qmv_mixbit_route(qbw_mixbit kind, const void* qp, const void* sc, const void* bi, int64_t group,
                            qbw_dtype xt, int64_t N, int64_t K, int* tensor_cores) {
    if (!tensor_cores) return QBW_EINVAL;
    size_t wbytes = 0;
    qbw_status st = mixbit_args(kind, qp, sc, bi, group, N, K, &wbytes);
    if (st != QBW_OK) return st;
    if (!valid_dtype(xt)) return QBW_EDTYPE;
    const int bits = (int)kind;
    const MixRoute r = mix_route(bits, sc, bi, group, xt, wbytes, K);
    if (!r.tc_form && !r.cuda_fits) return QBW_ESHAPE;
    DeviceInfo* di = nullptr;
    st = device_info(&di);
    if (st != QBW_OK) return st;
    CUtensorMap maps[3];
    const bool tc = mix_tc_maps(r, bits, qp, sc, bi, group, N, K, *di, maps);
    if (!tc && !r.cuda_fits) return QBW_ESHAPE;
    *tensor_cores = tc ? 1 : 0;
    return QBW_OK;
}

qbw_status qdequant_mixbit(qbw_mixbit kind, const void* qp, const void* sc, const void* bi, int64_t group, float* out,
                           int64_t N, int64_t K, void* stream) {
    size_t wbytes = 0;
    qbw_status st = mixbit_args(kind, qp, sc, bi, group, N, K, &wbytes);
    if (st != QBW_OK) return st;
    if (!out) return QBW_EINVAL;
    if ((uintptr_t)out % 4) return QBW_EALIGN;
    if (overlaps(out, (size_t)N * K * 4, qp, wbytes)) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaError_t e = launch_dequant_mixbit((int)kind, qp, sc, bi, (int)group, out, (int)N, (int)K, di->sm_count,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qbw_selftest_wait(int which, uint32_t limit_us, void* stream) {
    if (which < 0 || which > 1 || limit_us < 1 || limit_us > 2000000) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaError_t e = launch_selftest_wait(which, (uint64_t)limit_us * 1000ull, di->fault,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qdequant_q4_k(const void* w, float* out, int64_t N, int64_t K, void* stream) {
    return dequant_common(kFmtQ4K, w, out, N, K, stream);
}

qbw_status qdequant_q4_0(const void* w, float* out, int64_t N, int64_t K, void* stream) {
    return dequant_common(kFmtQ4, w, out, N, K, stream);
}

qbw_status qembed_q8_0(const void* w, const int32_t* ids, int64_t n_ids, void* out, qbw_dtype ot, int64_t N, int64_t K,
                       void* stream) {
    if (!w) return QBW_EINVAL;
    if (!valid_dtype(ot)) return QBW_EDTYPE;
    if (n_ids < 0 || n_ids > INT32_MAX || N < 1 || N > INT32_MAX || K < 32 || K % 32 != 0 || K > (int64_t(1) << 24))
        return QBW_ESHAPE;
    if (n_ids == 0) return QBW_OK;          // ids and out may be NULL
    if (!ids || !out) return QBW_EINVAL;
    if ((uintptr_t)ids % 4 || (uintptr_t)out % dtype_size(ot)) return QBW_EALIGN;
    const size_t obytes = (size_t)n_ids * (size_t)K * dtype_size(ot);
    if (overlaps(out, obytes, w, (size_t)N * (K / 32) * 34) || overlaps(out, obytes, ids, (size_t)n_ids * 4))
        return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaError_t e = launch_embed(kFmtQ8, static_cast<const uint8_t*>(w), ids, n_ids, N, K, out, ot == QBW_BF16,
                                 di->fault, di->sm_count, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qbw_chain_destroy(qbw_chain chain) {
    if (!chain) return QBW_EINVAL;
    int prev = -1;
    cudaGetDevice(&prev);
    bool ok = cudaSetDevice(chain->device) == cudaSuccess;
    ok = (!chain->steps || cudaFree(chain->steps) == cudaSuccess) && ok;
    ok = (!chain->bar || cudaFree(chain->bar) == cudaSuccess) && ok;
    ok = (!chain->share || cudaFree(chain->share) == cudaSuccess) && ok;
    if (prev >= 0) cudaSetDevice(prev);
    delete chain;
    return ok ? QBW_OK : QBW_ECUDA;
}

qbw_status qbw_chain_create(const qbw_chain_step* steps, int nsteps, qbw_chain* out) {
    if (!out) return QBW_EINVAL;
    *out = nullptr;
    if (!steps || nsteps < 1 || nsteps > (1 << 20)) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    const int ctas = qmv_chain_ctas(di->sm_count);
    if (ctas < 1) return QBW_ECUDA;
    std::vector<ChainStepDesc> host((size_t)nsteps);
    for (int i = 0; i < nsteps; ++i) {
        const qbw_chain_step& c = steps[i];
        if (!c.w || !c.x || !c.y) return QBW_EINVAL;
        if (!valid_dtype(c.yt)) return QBW_EDTYPE;
        const int nmat = c.w_up ? 2 : 1;
        if (c.N < 1 || c.N > INT32_MAX || c.K < 256 || c.K % 256 != 0 || c.K > (int64_t(1) << 24) ||
            !qmv_chain_step_supported(nmat, c.N, c.K, ctas))
            return QBW_ESHAPE;
        if ((uintptr_t)c.w % 16 || (uintptr_t)c.w_up % 16 || (uintptr_t)c.x % 16 || (uintptr_t)c.y % dtype_size(c.yt))
            return QBW_EALIGN;
        const size_t wbytes = (size_t)c.N * (size_t)weight_row_bytes(kFmtQ4, c.K);
        const size_t ybytes = (size_t)c.N * dtype_size(c.yt);
        if (overlaps(c.y, ybytes, c.x, (size_t)c.K * 2)) return QBW_EINVAL;
        for (int j = 0; j < nsteps; ++j) {     // no step writes weights
            const size_t wb = (size_t)steps[j].N * (size_t)weight_row_bytes(kFmtQ4, steps[j].K);
            if ((steps[j].w && overlaps(c.y, ybytes, steps[j].w, wb)) ||
                (steps[j].w_up && overlaps(c.y, ybytes, steps[j].w_up, wb)))
                return QBW_EINVAL;
        }
        ChainStepDesc& d = host[(size_t)i];
        std::memset(&d, 0, sizeof(d));
        if (!encode_q4_tile_map(&d.tmap[0], c.w, c.N, c.K) ||
            !encode_q4_tile_map(&d.tmap[1], nmat == 2 ? c.w_up : c.w, c.N, c.K))
            return QBW_ECUDA;
        qmv_chain_fill_step(&d, nmat, c.N, c.K);
        d.w[0] = static_cast<const uint8_t*>(c.w);
        d.w[1] = static_cast<const uint8_t*>(nmat == 2 ? c.w_up : c.w);
        d.x = c.x;
        d.y = c.y;
        d.y_bf16 = c.yt == QBW_BF16;
    }
    qbw_chain_s* ch = new qbw_chain_s;
    cudaGetDevice(&ch->device);
    ch->nsteps = nsteps;
    ch->ctas = ctas;
    ch->sm_count = di->sm_count;
    ch->host = host;
    ch->fault = di->fault;
    const size_t share_bytes = qmv_chain_share_bytes(ctas);
    if (cudaMalloc(&ch->steps, sizeof(ChainStepDesc) * (size_t)nsteps) != cudaSuccess ||
        cudaMalloc(&ch->bar, 2 * sizeof(unsigned int)) != cudaSuccess ||
        cudaMalloc(&ch->share, share_bytes) != cudaSuccess ||
        cudaMemcpy(ch->steps, host.data(), sizeof(ChainStepDesc) * (size_t)nsteps, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemset(ch->share, 0, share_bytes) != cudaSuccess || cudaMemset(ch->bar, 0, 2 * sizeof(unsigned int)) != cudaSuccess) {
        qbw_chain_destroy(ch);
        return QBW_ECUDA;
    }
    *out = ch;
    return QBW_OK;
}

qbw_status qbw_chain_run(qbw_chain chain, void* stream) {
    if (!chain) return QBW_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QBW_ECUDA;
    if (dev != chain->device) return QBW_EINVAL;
    cudaError_t e = launch_qmv_chain(chain->steps, chain->nsteps, chain->ctas, chain->bar, chain->share,
                                     chain->fault, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

qbw_status qbw_chain_run_launches(qbw_chain chain, void* stream) {
    if (!chain) return QBW_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return QBW_ECUDA;
    if (dev != chain->device) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < chain->nsteps; ++i) {
        const ChainStepDesc& d = chain->host[(size_t)i];
        if (!qmv_tc_supported(d.nmat, d.N, d.K, di->sm_count)) return QBW_ESHAPE;
    }
    for (int i = 0; i < chain->nsteps; ++i) {
        const ChainStepDesc& d = chain->host[(size_t)i];
        QtcNextLaunch next;
        next.units = 0;
        if (i + 1 < chain->nsteps) {
            const ChainStepDesc& n = chain->host[(size_t)i + 1];
            next.tmap[0] = n.tmap[0];
            next.tmap[1] = n.tmap[1];
            next.units = n.units;
            next.groups = n.groups;
            next.nmat = n.nmat;
        }
        const void* wp[2] = {d.w[0], d.w[1]};
        cudaError_t e = launch_qmv_tc(kFmtQ4, d.nmat, 1, d.tmap, wp, d.x, 1, d.y, d.y_bf16, d.N, d.K, di->sm_count,
                                      di->fault, s, &next);
        if (e != cudaSuccess) return QBW_ECUDA;
    }
    return QBW_OK;
}

qbw_status qbw_fault_read(uint32_t* code, int clear, void* stream) {
    if (!code) return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, di->fault, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return QBW_ECUDA;
    if (clear && cudaMemsetAsync(di->fault, 0, sizeof(unsigned int), s) != cudaSuccess) return QBW_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QBW_ECUDA;
    // a fault can leave split-K counters of the allocation-free entry point's
    // static scratch nonzero: its next call zero-fills the scratch again
    if (v != 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) noalloc_scratch_mark_dirty(dev);
    }
    *code = v;
    return QBW_OK;
}

}  // extern "C"
