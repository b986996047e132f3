// api.cu -- the C ABI of libqbw (include/qbw.h): argument validation, the
// per-device capability cache, the launch planner of the streaming kernels and
// the entry points themselves.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/qbw.h"
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

// Choose rows per task R, warps per CTA and ring depth for one streaming call.
// The model: every SM runs one CTA; time ~ (rounds of tasks per warp) x R rows,
// inflated by the activation reloads that small R pays, by an uneven final
// chunk, and by too few bytes in flight per SM or too few warps.
bool plan_stream(int fmt, int nmat, int64_t N, int64_t K, const DeviceInfo& di, StreamPlan* out) {
    const int64_t npairs = K / 64;
    const int nfull = (int)(npairs / 32);
    const int tail = (int)(npairs % 32);
    const size_t xs_bytes = (size_t)K * 4;
    const size_t fixed = align_up(xs_bytes, 128);
    const int Rs_1[] = {8, 4, 2, 1};
    const int Rs_2[] = {4, 2, 1};
    const int* Rs = (nmat == 2) ? Rs_2 : Rs_1;
    const int nR = (nmat == 2) ? 3 : 4;
    const int warp_opts[] = {16, 14, 12, 11, 10, 9, 8, 7, 6, 5, 4};
    double best = -1.0;
    for (int ir = 0; ir < nR; ++ir) {
        const int R = Rs[ir];
        const size_t stage = (size_t)nmat * R * chunk_bytes(fmt);
        const int64_t ntasks = (N + R - 1) / R;
        const double frac_tail = npairs ? (double)tail / (double)npairs : 0.0;
        double tail_eff = 1.0;
        if (tail) {
            const int items = R * tail;
            tail_eff = (double)items / (32.0 * (double)((items + 31) / 32));
        }
        const double k_eff = 1.0 / ((1.0 - frac_tail) + frac_tail / tail_eff);
        for (int w : warp_opts) {
            for (int depth = 4; depth >= 2; --depth) {
                const size_t ring = (size_t)w * depth * stage;
                const size_t bars = (size_t)w * depth * 8;
                const size_t smem = fixed + ring + bars;
                if (smem > di.smem_optin) continue;
                const int64_t P = (int64_t)di.sm_count * w;
                const int64_t rounds = (ntasks + P - 1) / P;
                const double eff = (double)ntasks / (double)(P * rounds);
                const double reuse = 1.0 / (1.0 + 0.12 / R);
                const double inflight = (double)w * (depth - 1) * (double)stage;
                const double lat = std::sqrt(std::min(1.0, inflight / 65536.0));
                const double occ = std::min(1.0, w / 8.0);
                const double score = eff * k_eff * reuse * lat * occ;
                if (score > best + 1e-9) {
                    best = score;
                    out->R = R;
                    out->warps = w;
                    out->depth = depth;
                    out->smem = smem;
                }
            }
        }
    }
    if (best < 0) return false;
    out->ctas = di.sm_count;
    StreamParams& p = out->p;
    p.row_bytes = (K / 32) * block_bytes(fmt);
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.npairs = (int32_t)npairs;
    p.ntasks = (int32_t)((N + out->R - 1) / out->R);
    p.nfull = nfull;
    p.tail_pairs = tail;
    p.depth = out->depth;
    p.ring_off = (uint32_t)fixed;
    p.stage_bytes = (uint32_t)((size_t)nmat * out->R * chunk_bytes(fmt));
    p.bar_off = (uint32_t)(fixed + (size_t)out->warps * out->depth * p.stage_bytes);
    p.fault = di.fault;
    return true;
}

int r_index(int R) { return R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3; }

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
    if ((uintptr_t)x % dtype_size(xt) || (uintptr_t)y % dtype_size(yt)) return QBW_EALIGN;
    const size_t wbytes = (size_t)N * (size_t)(K / 32) * block_bytes(fmt);
    const size_t ybytes = (size_t)N * dtype_size(yt);
    if (overlaps(y, ybytes, x, (size_t)K * dtype_size(xt)) || overlaps(y, ybytes, w0, wbytes) ||
        (nmat == 2 && overlaps(y, ybytes, w1, wbytes)))
        return QBW_EINVAL;
    DeviceInfo* di = nullptr;
    qbw_status st = device_info(&di);
    if (st != QBW_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool aligned = ((uintptr_t)w0 % 16 == 0) && (nmat == 1 || (uintptr_t)w1 % 16 == 0);
    if (K % 256 == 0 && aligned) {
        StreamPlan plan;
        if (plan_stream(fmt, nmat, N, K, *di, &plan)) {
            plan.p.w0 = static_cast<const uint8_t*>(w0);
            plan.p.w1 = static_cast<const uint8_t*>(nmat == 2 ? w1 : w0);
            plan.p.x = x;
            plan.p.y = y;
            plan.p.x_bf16 = (xt == QBW_BF16);
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

qbw_status qmv_gateup_q4_0(const void* w_gate, const void* w_up, const void* x, qbw_dtype xt, void* out,
                           qbw_dtype ot, int64_t M, int64_t N, int64_t K, void* stream) {
    return qmv_common(kFmtQ4, 2, w_gate, w_up, x, xt, out, ot, M, N, K, stream);
}

size_t qmm_q4_0_smallM_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

qbw_status qmm_q4_0_smallM(const void* w, const void* X, qbw_dtype xt, void* Y, qbw_dtype yt, int64_t M,
                           int64_t N, int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
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
    cudaError_t e = launch_qmm_generic(static_cast<const uint8_t*>(w), X, Y, yt == QBW_BF16, M, N, K, di->sm_count,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QBW_OK : QBW_ECUDA;
}

static qbw_status dequant_common(int fmt, const void* w, float* out, int64_t N, int64_t K, void* stream) {
    if (!w || !out) return QBW_EINVAL;
    if (N < 1 || K < 32 || K % 32 != 0 || K > (int64_t(1) << 24) || N > INT32_MAX) return QBW_ESHAPE;
    if ((uintptr_t)out % 4) return QBW_EALIGN;
    if (overlaps(out, (size_t)N * K * 4, w, (size_t)N * (K / 32) * block_bytes(fmt))) return QBW_EINVAL;
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

qbw_status qdequant_q4_0(const void* w, float* out, int64_t N, int64_t K, void* stream) {
    return dequant_common(kFmtQ4, w, out, N, K, stream);
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
    *code = v;
    return QBW_OK;
}

}  // extern "C"
